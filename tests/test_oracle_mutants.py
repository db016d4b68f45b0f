"""The pins must bite: each planted mistake in a copy of the oracle's C source
(a dropped term, a wrong index, a sign, a wrong rounding, a missing reset, an
inclusive-for-exclusive prefix) has to make at least one pin fail.

Mistakes are planted in a temporary copy of the source, on the CPU, never in
the oracle that the other tests use.
"""
import os

import pytest

import oracle_pins
from oracle import Oracle, load
from oracle.oracle import _SRC, compile_library

CPLX_FWD_STEP = 'STATE xr = LOAD(ar[i]), xi = LOAD(ai[i]);                      \\\n                STATE nr = FMA(xr, hr, FMA(-xi, hi, LOAD(br[i])));             \\\n                STATE ni = FMA(xi, hr, FMA(xr, hi, LOAD(bi[i])));'

MUTANTS = {
    "fwd_f64_drops_b": ("h[d] = fma(a[i], h[d], b[i]);", "h[d] = a[i] * h[d];"),
    "fwd_f64_no_row_reset": ("for (int64_t d = 0; d < D; ++d) h[d] = 0.0;\n", "\n"),
    "fwd_f32_two_roundings": ("h[d] = fmaf(a[i], h[d], b[i]);", "h[d] = a[i] * h[d] + b[i];"),
    "bwd_f64_uses_a_t": ("g[d] = fma(a[i + D], g[d], grad_out[i]);",
                         "g[d] = fma(a[i], g[d], grad_out[i]);"),
    "bwd_f64_uses_h_t": ("double h_prev = (t > 0) ? out[i - D] : 0.0;",
                         "double h_prev = out[i];"),
    "bwd_f64_sign": ("grad_a[i] = g[d] * h_prev;\n            }\n        }\n    }\n    free(g);\n"
                     "    return LRO_OK;\n}\n\n/* ---",
                     "grad_a[i] = -g[d] * h_prev;\n            }\n        }\n    }\n    free(g);\n"
                     "    return LRO_OK;\n}\n\n/* ---"),
    "bwd_f32_drops_carry": ("g[d] = fmaf(a[i + D], g[d], grad_out[i]); /* a_{t+1} */",
                            "g[d] = grad_out[i];"),
    "bf16_round_half_up": ("u += 0x7fffu + keep_lsb;", "u += 0x8000u;"),
    "bf16_bwd_prev_from_state": ("float h_prev = (t > 0) ? lro_bf16_to_f32(out[i - D]) : 0.0f;",
                                 "float h_prev = (t > 0) ? lro_bf16_to_f32(out[i]) : 0.0f;"),
    "chunk_prefix_inclusive": ("hin[c] = state;                                                \\\n"
                               "                state = FMA(P[c], state, Q[c]);",
                               "state = FMA(P[c], state, Q[c]);                                \\\n"
                               "                hin[c] = state;"),
    "chunk_reverse_summary_drops_direct": ("k = a[i] * k + a[i] * grad_out[i];", "k = a[i] * k;"),
    "state_fwd_ignores_h0": ("STATE h = h0 ? h0[bb * D + d] : 0;", "STATE h = 0;"),
    "state_fwd_ignores_resets": ("STATE x = resets(seg, bb, T, t) ? 0 : LOAD(a[i]);", "STATE x = LOAD(a[i]);"),
    "state_bwd_reset_on_wrong_step": ("(resets(seg, bb, T, t + 1) ? 0 : LOAD(a[i + D]))",
                                      "(resets(seg, bb, T, t) ? 0 : LOAD(a[i + D]))"),
    "state_bwd_drops_grad_last": ("STATE g = grad_last ? grad_last[bb * D + d] : 0;", "STATE g = 0;"),
    "state_bwd_prev_ignores_h0": (": (h0 ? h0[bb * D + d] : 0);", ": 0;"),
    "state_grad_h0_drops_decay": ("? 0 : LOAD(a[bb * T * D + d]) * g;", "? 0 : g;"),
    "state_grad_a_not_masked": ("grad_a[i] = resets(seg, bb, T, t) ? STORE(0) : STORE(g * h_prev);",
                                "grad_a[i] = STORE(g * h_prev);"),
    "state_grad_h0_ignores_first_reset": ("grad_h0[bb * D + d] = resets(seg, bb, T, 0)",
                                          "grad_h0[bb * D + d] = 0"),
    "state_empty_grad_h0_zero": ("grad_h0[bb * D + d] = g;", "grad_h0[bb * D + d] = 0;"),
    # anchors include the plain complex body's own loads (the state-carrying
    # complex body repeats these statements)
    "complex_fwd_sign": (CPLX_FWD_STEP, CPLX_FWD_STEP.replace("FMA(-xi, hi, LOAD(br[i]))", "FMA(xi, hi, LOAD(br[i]))")),
    "complex_fwd_swapped_parts": (CPLX_FWD_STEP, CPLX_FWD_STEP.replace("FMA(xi, hr, FMA(xr, hi, LOAD(bi[i])))",
                                                                       "FMA(xi, hi, FMA(xr, hr, LOAD(bi[i])))")),
    "complex_bwd_no_conjugate": ("                    STATE ni = FMA(xr, gi, FMA(-xi, gr, yi));",
                                 "                    STATE ni = FMA(xr, gi, FMA(xi, gr, yi));"),
    "complex_bwd_uses_a_t": ("STATE xr = LOAD(ar[i + D]), xi = LOAD(ai[i + D]);",
                             "STATE xr = LOAD(ar[i]), xi = LOAD(ai[i]);"),
    "complex_grad_a_not_conjugated": ("\n                grad_ai[i] = STORE(FMA(gi, pr, -(gr * pi)));",
                                      "\n                grad_ai[i] = STORE(FMA(gi, pr, gr * pi));"),
    "complex_grad_a_drops_cross_term": ("\n                grad_ar[i] = STORE(FMA(gr, pr, gi * pi));",
                                        "\n                grad_ar[i] = STORE(gr * pr);"),
    "cstate_fwd_ignores_h0": ("STATE hr = h0_r ? h0_r[bb * D + d] : 0;", "STATE hr = 0;"),
    "cstate_fwd_ignores_resets": ("STATE xr = r ? 0 : LOAD(ar[i]), xi = r ? 0 : LOAD(ai[i]);",
                                  "STATE xr = LOAD(ar[i]), xi = LOAD(ai[i]);"),
    "cstate_bwd_drops_grad_last": ("STATE gr = gl_r ? gl_r[bb * D + d] : 0;", "STATE gr = 0;"),
    "cstate_bwd_reset_on_wrong_step": ("} else if (resets(seg, bb, T, t + 1)) {", "} else if (resets(seg, bb, T, t)) {"),
    "cstate_bwd_prev_ignores_h0": ("LOAD(out_i[i - D]) : (h0_i ? h0_i[bb * D + d] : 0)", "LOAD(out_i[i - D]) : 0"),
    "cstate_grad_a_not_masked": ("grad_ai[i] = STORE(0);", "grad_ai[i] = STORE(FMA(gi, pr, -(gr * pi)));"),
    "cstate_grad_h0_not_conjugated": ("hi = FMA(xr, gi, -(xi * gr));", "hi = FMA(xr, gi, xi * gr);"),
    "gated_rate_sign": ("STATE la = -(nu * e);                                          \\\n                h = FMA",
                        "STATE la = nu * e;                                             \\\n                h = FMA"),
    "gated_bwd_rate_not_exponentiated": ("STATE nu = EXP(nu_log[d]);                                         \\\n            STATE g = 0",
                                         "STATE nu = nu_log[d];                                              \\\n            STATE g = 0"),
    "gated_q_drops_decay": ("STATE q = (grad_a * a) * la;", "STATE q = grad_a * la;"),
    "gated_nu_overwrites": ("acc_nu[d] += (double)q;", "acc_nu[d] = (double)q;"),
    "gated_carry_uses_a_t": (": FMA(a_next, g, LOAD(grad_out[i]));", ": FMA(a, g, LOAD(grad_out[i]));"),
}


def _run_all_pins(o):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        if pin.__name__ == "pin_symbolic_small_T":
            try:
                import sympy  # noqa: F401
            except ImportError:
                continue
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(_SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique in the oracle source"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    so = compile_library(str(mutant_src), str(tmp_path / "libmutant.so"))
    failed = _run_all_pins(Oracle(load(so)))
    assert failed, f"no pin caught the planted mistake {name}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    so = compile_library(_SRC, str(tmp_path / "libcopy.so"))
    assert _run_all_pins(Oracle(load(so))) == []
