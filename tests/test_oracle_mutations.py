"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of oracle.c (on the CPU), builds it
and runs the pin suite against it in a subprocess: the suite must fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "skip_sign_flipped": ("(c < ln_lambda)", "(c > ln_lambda)"),
    "vote_min_not_max": ("if (diff > c) c = diff;", "if (c == -INFINITY || diff < c) c = diff;"),
    "l_not_rescaled": ("st->l[r] *= alpha;", ""),
    "alpha_sign": ("exp(st->m[r] - m_new)", "exp(m_new - st->m[r])"),
    "gqa_head_map": ("kvh = h / G;", "kvh = h % p->Hkv;"),
    "causal_top_left": ("row + off : (int64_t)p->Lk - 1", "row : (int64_t)p->Lk - 1"),
    "scale_dropped": ("x = scale * dot_bf16", "x = dot_bf16"),
    "merge_weight_sign": ("exp(sm[(size_t)g * S + sp] - mstar)", "exp(mstar - sm[(size_t)g * S + sp])"),
    "split_floor": ("T = ceil_div(nT, S)", "T = (nT / S > 0 ? nT / S : 1)"),
    "calib_edge": ("a = L * exp(0.5 * (lo + hi));", "a = L * exp(lo);"),
    "value_head_stride_key_width": ("* p->Lk * dk;\n    const uint16_t* vh = v + (size_t)(b * p->Hkv + kvh) * p->Lk * d;",
                                    "* p->Lk * dk;\n    const uint16_t* vh = v + (size_t)(b * p->Hkv + kvh) * p->Lk * dk;"),
    "value_row_stride_key_width": ("vh + (size_t)(k0 + t) * d;", "vh + (size_t)(k0 + t) * dk;"),
    "v_transposed": ("p * bf16_to_double(vk[e])", "p * bf16_to_double(vh[(size_t)e * d + (k0 + t) % d])"),
    "O_not_rescaled": ("for (int e = 0; e < d; ++e) Or[e] *= alpha;", ""),
    "tie_skips": ("(c < ln_lambda)", "(c <= ln_lambda)"),
    "masked_row_vetoes": ("if (tmax[r] == -INFINITY) continue; /* no visible key: no veto */", ""),
    "not_evaluated_counted_as_skipped": ("*c_out = NAN;\n    return ORC_NOT_EVALUATED;",
                                         "*c_out = NAN;\n    return ORC_SKIPPED;"),
    "causal_diagonal_excluded": ("row + off : (int64_t)p->Lk - 1", "row + off - 1 : (int64_t)p->Lk - 1"),
    "calib_floor_not_round": ("floor(target * (double)N + 0.5)", "floor(target * (double)N)"),
    "calib_unreachable_gives_zero": ("      a = L;\n", "      a = 0.0;\n"),
    "causal_mask_ignored": ("if (key <= last_visible[r]) x = scale", "x = scale"),
    "margin_after_update": ("const double diff = (st->m[r] == -INFINITY) ? INFINITY : tmax[r] - st->m[r];",
                            "const double diff = (st->m[r] == -INFINITY) ? INFINITY : "
                            "tmax[r] - (tmax[r] > st->m[r] ? tmax[r] : st->m[r]);"),
    "split_state_carried_over": ("      /* Each split runs its own online pass from an empty state. */\n"
                                 "      state_reset(&st);", "      if (sp == 0) state_reset(&st);"),
    "merge_l_unweighted": ("l += ls * w;", "l += ls;"),
    "split_size_floor_plus_one": ("T = ceil_div(nT, S)", "T = nT / S + 1"),
    "decode_heads_interleaved": ("q + ((size_t)b * p->Hq + (size_t)kvh * G + g) * dk;",
                                 "q + ((size_t)b * p->Hq + (size_t)g * p->Hkv + kvh) * dk;"),
    "calib_lambda_above_one": ("if (hi > 0.0) hi = 0.0; /* lambda <= 1 */", ""),
    # prefill with value rows of another width than query/key rows
    "prefill_query_rows_value_width": ("(size_t)row) * dk;", "(size_t)row) * d;"),
    "prefill_output_rows_key_width": ("double* ou = o + (size_t)i * Bq * d;\n      memset(ou, 0, sizeof(double) * (size_t)Bq * d);",
                                      "double* ou = o + (size_t)i * Bq * dk;\n      memset(ou, 0, sizeof(double) * (size_t)Bq * d);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mutation(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = tmp_path / "oracle.c"
    mutated.write_text(src.replace(old, new))
    (tmp_path / "oracle.h").write_text(open(os.path.join(ROOT, "oracle", "oracle.h")).read())
    lib = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(lib),
                           str(mutated), "-lm"])
    env = dict(os.environ, SSATTN_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutation {name} survived the pins:\n{r.stdout[-2000:]}"
