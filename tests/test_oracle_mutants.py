"""Plant plausible mistakes in a copy of oracle.c and check that each one
fails at least one pin of tests/test_oracle.py.

The mutated copies are compiled into a temporary directory; the oracle's own
source and library are never touched.  This is how the pins are shown to be
sharp enough: a dropped term, a wrong sign or index, a transposed operand or a
missing -inf guard each break some page-printed value, closed form, invariant
or library special case.
"""
import inspect
import os
import shutil

import pytest

import oracle
from oracle import build as obuild
import tests.test_oracle as pins

if shutil.which("gcc") is None:  # pragma: no cover
    pytest.skip("gcc not available", allow_module_level=True)

# (name, original text, mutated text): each original must occur exactly once.
MUTANTS = [
    ("drop_scale", "s[j] = scale * acc;", "s[j] = acc;"),
    ("mask_off_by_one", "if (j > last_visible ||", "if (j >= last_visible ||"),
    ("window_left_ignored", "if (j > last_visible || j < first_visible) {", "if (j > last_visible) {"),
    ("window_left_off_by_one", "first_visible = job->wl < 0 ? 0 : i + off - job->wl;",
     "first_visible = job->wl < 0 ? 0 : i + off - job->wl + 1;"),
    ("window_right_off_by_one", "last_visible = job->wr < 0 ? job->nk - 1 : i + off + job->wr;",
     "last_visible = job->wr < 0 ? job->nk - 1 : i + off + job->wr + 1;"),
    ("causal_offset_sign", "i + (job->nk - job->nq)", "i - (job->nk - job->nq)"),
    ("k_feature_index", "qi[c] * k[j * d + c]", "qi[c] * k[j * d + (d - 1 - c)]"),
    ("v_feature_index", "oi[c] += p * v[j * d + c];", "oi[c] += p * v[j * d + (d - 1 - c)];"),
    ("pass3_no_max", "double p = exp(s[j] - m) / l;", "double p = exp(s[j]) / l;"),
    ("pass2_no_max", "l += exp(s[j] - m);", "l += exp(s[j]);"),
    ("lse_no_max", "*lse_i = m + log(l);", "*lse_i = log(l);"),
    ("max_init_zero", "double m = -INFINITY;\n    for (int64_t j = 0; j < nk; ++j)",
     "double m = 0.0;\n    for (int64_t j = 0; j < nk; ++j)"),
    ("no_masked_row_case", "if (m == -INFINITY) {\n        for (int64_t c = 0; c < d; ++c)\n            oi[c] = 0.0;",
     "if (0) {\n        for (int64_t c = 0; c < d; ++c)\n            oi[c] = 0.0;"),
    ("online_no_o_rescale", "o[c] = o[c] * alpha;", "o[c] = o[c];"),
    ("online_no_l_rescale", "l = l * alpha;", "l = l;"),
    ("online_alpha_sign", "double alpha = exp(m - ref);", "double alpha = exp(ref - m);"),
    ("online_p_old_max", "double p = exp(s[j] - ref);", "double p = exp(s[j] - m);"),
    ("online_no_inf_guard", "double ref = (m_new == -INFINITY) ? 0.0 : m_new;\n        double alpha",
     "double ref = m_new;\n        double alpha"),
    ("online_max_not_kept", "        m = m_new;\n    }\n\n    *m_out = m;", "    }\n\n    *m_out = m;"),
    ("merge_weight_no_exp", "double w1 = (m1 == -INFINITY) ? 0.0 : l1 * exp(m1 - mm);",
     "double w1 = (m1 == -INFINITY) ? 0.0 : l1;"),
    ("merge_weights_swapped", "o_out[c] * (w1 / ll) + o2[c] * (w2 / ll)",
     "o_out[c] * (w2 / ll) + o2[c] * (w1 / ll)"),
    ("merge_lse_no_max", "*lse_out = (l1 == 0.0) ? -INFINITY : m1 + log(l1);",
     "*lse_out = (l1 == 0.0) ? -INFINITY : log(l1);"),
    ("two_pass_no_rescale", "l = exp(m - ref) * l + exp(x[i] - ref);", "l = l + exp(x[i] - ref);"),
    ("softmax_rows_selection_ignored", "oracle_softmax_two_pass(job->x + i * job->cols,",
     "oracle_softmax_two_pass(job->x + r * job->cols,"),
    ("fp8_k_feature_index", "t += k[j * d + c] * qi[c];", "t += k[j * d + (d - 1 - c)] * qi[c];"),
    ("fp8_lse_no_max", "*lse_i = log(l) + m;", "*lse_i = log(l);"),
    ("fp8_no_sum_scale", "    l *= 1.0 / 256.0; /* sum_scale */", "    /* l not rescaled */"),
    ("fp8_no_final_scale", "const double final_scale = v_descale / 256.0;", "const double final_scale = v_descale;"),
    ("fp8_no_quantisation", "double p8 = oracle_e4m3(pp);", "double p8 = pp;"),
    ("fp8_acc_not_rescaled", "        acc[c] *= alpha;\n", "        acc[c] *= 1.0;\n"),
    ("fp8_no_max_offset", "double pp = exp2((s[j] - m_new) * log2e + 8.0);", "double pp = exp2((s[j] - m_new) * log2e);"),
    ("e4m3_ties_away", "double r = nearbyint(a / spacing) * spacing;", "double r = round(a / spacing) * spacing;"),
    ("bwd_dq_no_scale", "dqi[c] += J->scale * ds * J->k[j * d + c];", "dqi[c] += ds * J->k[j * d + c];"),
    ("bwd_dk_wrong_operand", "dkj[c] += J->scale * ds * J->q[i * d + c];",
     "dkj[c] += J->scale * ds * J->k[j * d + c];"),
    ("bwd_dv_wrong_operand", "dvj[c] += p * J->dout[i * d + c];", "dvj[c] += p * J->v[j * d + c];"),
    ("bwd_D_without_p", "di += p * dot(J->dout + i * d, J->v + j * d, d);",
     "di += dot(J->dout + i * d, J->v + j * d, d);"),
    ("bwd_p_without_scale", "return exp(J->scale * dot(J->q + i * J->d, J->k + j * J->d, J->d) - J->lse[i]);",
     "return exp(dot(J->q + i * J->d, J->k + j * J->d, J->d) - J->lse[i]);"),
    ("softmax_rows_skips_a_row", "for (int64_t r = job->r_begin; r < job->r_end; ++r) {\n        int64_t i = job->sel",
     "for (int64_t r = job->r_begin + 1; r < job->r_end; ++r) {\n        int64_t i = job->sel"),
]


def _pin_calls():
    """Every pin in tests/test_oracle.py, with one representative argument set."""
    golden = pins.golden.__wrapped__() if hasattr(pins.golden, "__wrapped__") else None
    if golden is None:
        import json
        with open(pins.GOLDEN, encoding="utf-8") as f:
            golden = json.load(f)
    params = {
        "test_attention_matches_scipy_softmax": [(5, 7, 3, False, 0), (4, 9, 2, True, 2), (9, 4, 3, True, 3)],
        "test_zero_queries_average_visible_values": [(False,), (True,)],
        "test_online_blocks_match_three_pass": [(0,)],
        "test_merge_of_random_partition_matches_full": [(0,)],
        "test_window_matches_scipy_softmax": [(10, 10, 2, 0, 0), (6, 14, 4, 1, 2), (14, 6, 0, 2, 3)],
        "test_bwd_matches_finite_differences": [(3, 4, 2, (-1, -1), 0), (4, 6, 2, (1, 1), 3)],
        "test_fp8_exact_when_every_p_is_representable": [(False,), (True,)],
    }
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        sig = inspect.signature(fn)
        if "golden" in sig.parameters:
            calls.append((name, lambda fn=fn: fn(golden)))
        elif name in params:
            for args in params[name]:
                calls.append((f"{name}{args}", lambda fn=fn, a=args: fn(*a)))
        elif not sig.parameters:
            calls.append((name, fn))
    return calls


def test_every_pin_passes_on_the_real_oracle():
    for name, call in _pin_calls():
        call()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, monkeypatch, name, old, new):
    with open(obuild.SRC, encoding="utf-8") as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/present"
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(src.replace(old, new), encoding="utf-8")
    lib_path = obuild.compile_oracle(str(mutated), str(tmp_path / "liboracle_mutant.so"), werror=False)
    monkeypatch.setattr(oracle, "_lib", oracle.load(lib_path))
    failed = []
    for pin, call in _pin_calls():
        try:
            call()
        except Exception:  # AssertionError, or a NaN tripping numpy's checks
            failed.append(pin)
    assert failed, f"mutant {name} survived every pin"
