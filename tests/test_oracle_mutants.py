"""The pins must be able to fail: plant plausible mistakes in a copy of the
oracle's C source (on the CPU), rebuild it, and check that the pin suite
rejects every mutant."""
import ctypes
import os
import subprocess

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "oracle.c")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("drop_scale", "double s = p->scale * acc;", "double s = acc;"),
    ("gqa_modulo", "const long g = h / (p->Hq / p->Hkv);", "const long g = h % p->Hkv;"),
    ("mask_off_by_one", "long end = (p->causal == 1) ? i + (p->Skv - p->Sq) + 1 : i + 1;",
     "long end = (p->causal == 1) ? i + (p->Skv - p->Sq) : i;"),
    ("bottom_right_as_top_left", "long end = (p->causal == 1) ? i + (p->Skv - p->Sq) + 1 : i + 1;",
     "long end = i + 1;"),
    ("top_left_as_bottom_right", "long end = (p->causal == 1) ? i + (p->Skv - p->Sq) + 1 : i + 1;",
     "long end = i + (p->Skv - p->Sq) + 1;"),
    ("base2_lse", "= m + log(l);", "= m + log2(l);"),
    ("no_normalise", "for (long d = 0; d < D; ++d) o[d] /= l;", ";"),
    ("exp2_weights", "double w = exp(s_buf[j - j_lo] - m);", "double w = exp2(s_buf[j - j_lo] - m);"),
    ("no_max_shift", "double w = exp(s_buf[j - j_lo] - m);", "double w = exp(s_buf[j - j_lo]);"),
    ("k_by_query_row", "const uint16_t *krow = p->k + ((b * p->Skv + j) * p->Hkv + g) * D;",
     "const uint16_t *krow = p->k + ((b * p->Skv + (i < p->Skv ? i : j)) * p->Hkv + g) * D;"),
    ("k_head_modulo", "const uint16_t *krow = p->k + ((b * p->Skv + j) * p->Hkv + g) * D;",
     "const uint16_t *krow = p->k + ((b * p->Skv + j) * p->Hkv + h % p->Hkv) * D;"),
    ("v_by_query_row", "const uint16_t *vrow = p->v + ((b * p->Skv + j) * p->Hkv + g) * D;",
     "const uint16_t *vrow = p->v + ((b * p->Skv + (i < p->Skv ? i : j)) * p->Hkv + g) * D;"),
    ("sign_flip", "double s = p->scale * acc;", "double s = -p->scale * acc;"),
    ("f16_read_as_bf16", "return p->f16 ? widen_f16(bits) : widen_bf16(bits);",
     "return widen_bf16(bits);"),
    ("f16_exponent_bias", "mag = ldexp((double)(1024 + frac), e - 25);",
     "mag = ldexp((double)(1024 + frac), e - 24);"),
    ("f16_subnormal_scale", "mag = ldexp((double)frac, -24); /* zero and subnormals */",
     "mag = ldexp((double)frac, -25);"),
    # backward
    ("bwd_dq_no_scale", "dq[d] *= p->scale;", ";"),
    ("bwd_delta_sign", "ds_buf[j] = p_buf[j] * (ds_buf[j] - delta);",
     "ds_buf[j] = p_buf[j] * (ds_buf[j] + delta);"),
    ("bwd_no_delta", "ds_buf[j] = p_buf[j] * (ds_buf[j] - delta);",
     "ds_buf[j] = p_buf[j] * ds_buf[j];"),
    ("bwd_unnormalised_weights", "p_buf[j] = exp(p_buf[j] - lse);", "p_buf[j] = exp(p_buf[j] - m);"),
    ("bwd_dv_from_ds", "dv[d] += p_buf[j] * dod[d];", "dv[d] += ds_buf[j] * dod[d];"),
    ("bwd_dk_from_do", "dk[d] += scale * ds_buf[j] * qd[d];", "dk[d] += scale * ds_buf[j] * dod[d];"),
    ("bwd_dk_no_scale", "dk[d] += scale * ds_buf[j] * qd[d];", "dk[d] += ds_buf[j] * qd[d];"),
    ("bwd_dp_from_q", "dp += dod[d] * widen(p, vrow[d]);", "dp += qd[d] * widen(p, vrow[d]);"),
    ("bwd_dq_from_p", "dq[d] += ds_buf[j] * widen(p, krow[d]);",
     "dq[d] += p_buf[j] * widen(p, krow[d]);"),
    ("bwd_strided_group", "for (long h = g * G; h < (g + 1) * G; ++h)",
     "for (long h = g; h < Hq; h += Hkv)"),
    ("bwd_keys_base2", "const double pij = exp(scale * s - lse[hi]);",
     "const double pij = exp2(scale * s - lse[hi]);"),
    ("bwd_keys_delta_sign", "const double ds = pij * (dp - delta[hi]);",
     "const double ds = pij * (dp + delta[hi]);"),
    ("bwd_keys_mask_off_by_one", "if (j >= visible_end(&p, i)) continue;",
     "if (j > visible_end(&p, i)) continue;"),
    ("bwd_supplied_delta_ignored", "if (delta_in) delta = delta_in[(b * p->Hq + h) * p->Sq + i];", ";"),
    ("bwd_supplied_delta_row_major", "if (delta_in) delta = delta_in[(b * p->Hq + h) * p->Sq + i];",
     "if (delta_in) delta = delta_in[(b * p->Sq + i) * p->Hq + h];"),
    ("bwd_keys_supplied_delta_ignored", "delta[hi] = delta_in ? delta_in[(b * Hq + h) * Sq + i] : dl;",
     "delta[hi] = dl;"),
]

PIN_TESTS = [
    "test_hand_worked_two_keys", "test_zero_query_closed_form", "test_constant_v_rows",
    "test_causal_row0_is_v0", "test_one_hot_limit_pins_operand_roles", "test_matches_scipy_softmax",
    "test_brute_force_twin", "test_gqa_head_repeat_equivalence",
    "test_bottom_right_equals_tail_of_square_causal", "test_shift_invariance_large_logits",
    "test_merge_identity_random_chunks", "test_top_left_rules",
    "test_f16_widening_every_finite_pattern", "test_f16_brute_force_twin",
]

BWD_PIN_TESTS = [
    "test_bwd_finite_differences", "test_bwd_matches_torch_autograd",
    "test_bwd_hand_worked_two_keys", "test_bwd_zero_query_closed_form",
    "test_bwd_constant_values_give_zero_dq_dk", "test_bwd_invariants",
    "test_bwd_gqa_equals_repeated_heads", "test_bwd_sampled_entry_points_match_full",
    "test_bwd_fully_masked_rows_contribute_nothing", "test_bwd_supplied_delta_equal_to_exact",
    "test_bwd_delta_shift",
]


def _build_mutant(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation anchor for {name} not found"
    src = tmp_path / f"{name}.c"
    src.write_text(text.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-std=c11", str(src), "-o",
                    str(so), "-lm"], check=True)
    return oracle.configure(ctypes.CDLL(str(so)))


def _run_pins(monkeypatch, lib):
    import test_oracle_bwd_pins as bwd_pins
    import test_oracle_pins as pins
    monkeypatch.setattr(oracle, "_lib", lib)
    failures = 0
    for module, name in [(pins, n) for n in PIN_TESTS] + [(bwd_pins, n) for n in BWD_PIN_TESTS]:
        fn = getattr(module, name)
        params = getattr(fn, "pytestmark", [])
        cases = [dict()]
        for mark in params:
            if mark.name == "parametrize":
                argnames = [a.strip() for a in mark.args[0].split(",")] if isinstance(
                    mark.args[0], str) else list(mark.args[0])
                new_cases = []
                for c in cases:
                    for val in mark.args[1]:
                        vals = val if len(argnames) > 1 else (val,)
                        new_cases.append({**c, **dict(zip(argnames, vals))})
                cases = new_cases
        for kw in cases:
            try:
                fn(**kw)
            except (AssertionError, ValueError, FloatingPointError):
                failures += 1
    return failures


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_planted_mistake(tmp_path, monkeypatch, name, old, new):
    import sys
    sys.path.insert(0, HERE)
    lib = _build_mutant(tmp_path, name, old, new)
    assert _run_pins(monkeypatch, lib) > 0, f"mutant {name} passed every pin"


def test_unmutated_copy_passes(tmp_path, monkeypatch):
    import sys
    sys.path.insert(0, HERE)
    lib = _build_mutant(tmp_path, "identity", "int oracle_num_threads(void)",
                        "int oracle_num_threads(void)")
    assert _run_pins(monkeypatch, lib) == 0
