"""Plant plausible mistakes in copies of the oracle source and check that
each broken copy fails at least one pin.  This is what makes the pins worth
trusting: a dropped term, a wrong sign, a swapped operand or a wrong rounding
anywhere in the oracle would be caught."""
import os

import pytest

import oracle
import oracle_pins as P

# (name, exact text in adamw_ref.c, replacement)
MUTANTS = [
    ("no_weight_decay_bf16", "float upd = (s.step_size * (ms / den)) + (s.lrwd * p0);",
     "float upd = (s.step_size * (ms / den));"),
    ("no_weight_decay_mixed", "float upd = (s.step_size * (m1 / den)) + (s.lrwd * p0);",
     "float upd = (s.step_size * (m1 / den));"),
    ("update_sign", "float y = c0 - upd;", "float y = c0 + upd;"),
    ("mixed_update_sign", "float pn = p0 - upd;", "float pn = p0 + upd;"),
    ("no_bias_correction1", "s.step_size = (float)((double)hp->lr / bc1);",
     "s.step_size = (float)((double)hp->lr); (void)bc1;"),
    ("no_bias_correction2", "s.sbc2 = (float)sqrt(bc2);", "s.sbc2 = 1.0f; (void)bc2;"),
    ("bc2_uses_beta1", "double bc2 = 1.0 - power_by_squaring(b2, t);",
     "double bc2 = 1.0 - power_by_squaring(b1, t);"),
    ("power_off_by_one", "    double result = 1.0, square = b;\n",
     "    double result = b, square = b;\n"),
    ("power_skips_odd_bits", "        if (t & 1) result = result * square;\n",
     "        if (t & 2) result = result * square;\n"),
    ("v_not_squared_mixed", "float v1 = (b2 * v[i]) + ((s.omb2 * gi) * gi);",
     "float v1 = (b2 * v[i]) + (s.omb2 * gi);"),
    ("v_not_squared_bf16", "float v1 = (b2 * v0) + ((s.omb2 * gi) * gi);",
     "float v1 = (b2 * v0) + ((s.omb2 * gi) * fabsf(gi) * 0.5f);"),
    ("betas_swapped_mixed", "float m1 = (b1 * m[i]) + (s.omb1 * gi);",
     "float m1 = (b2 * m[i]) + (s.omb1 * gi);"),
    ("betas_swapped_bf16", "float m1 = (b1 * m0) + (s.omb1 * gi);",
     "float m1 = (b2 * m0) + (s.omb1 * gi);"),
    ("eps_dropped_mixed", "float den = (sqrtf(v1) / s.sbc2) + eps;",
     "float den = (sqrtf(v1) / s.sbc2);"),
    ("eps_inside_sqrt_bf16", "float den = (sqrtf(vs) / s.sbc2) + eps;",
     "float den = (sqrtf(vs + eps) / s.sbc2);"),
    ("kahan_comp_sign", "uint16_t cnh = f32_to_bf16_rne(y - (pn - p0));",
     "uint16_t cnh = f32_to_bf16_rne(y + (pn - p0));"),
    ("kahan_ignores_c", "uint16_t pnh = f32_to_bf16_rne(p0 + y);",
     "uint16_t pnh = f32_to_bf16_rne(p0 - upd);"),
    ("kahan_c_not_updated", "        c[i] = cnh;\n", "        (void)cnh;\n"),
    ("bf16_truncates", "    u += 0x7fffu + keep_lsb;\n", "    (void)keep_lsb;\n"),
    ("bf16_ties_away", "    u += 0x7fffu + keep_lsb;\n", "    u += 0x8000u; (void)keep_lsb;\n"),
    ("moments_unrounded_bf16", "float ms = bf16_bits_to_f32(m1h);", "float ms = m1 * 1.01f;"),
    ("pout_from_old_master", "p_out[i] = f32_to_bf16_rne(pn);", "p_out[i] = f32_to_bf16_rne(p0);"),
    ("norm_no_sqrt", "double norm = sqrt(sumsq);", "double norm = sumsq;"),
    ("clip_not_clamped", "if (coef > 1.0) coef = 1.0;", "(void)0;"),
    ("clip_no_eps", "double coef = (double)max_norm / (norm + 1e-6);",
     "double coef = (double)max_norm / (norm);"),
    ("norm_abs_not_square", "double sq = x * x;", "double sq = fabs(x);"),
    ("norm_uncompensated", "    acc[1] = comp;\n", "    acc[1] = 0.0 * comp;\n"),
    ("nonfinite_missed", "if (!isfinite(x)) bad = 1;", "(void)0;"),
    ("skip_still_writes", "        if (bad) return 1;\n", "        (void)bad;\n"),
    ("split_truncates", "    uint16_t hi = (uint16_t)((u + 0x8000u) >> 16);\n",
     "    uint16_t hi = (uint16_t)(u >> 16);\n"),
    ("join_ignores_remainder", "    uint32_t u = ((uint32_t)p16 << 16) + (uint32_t)(int32_t)r16;\n",
     "    uint32_t u = ((uint32_t)p16 << 16); (void)r16;\n"),
    ("remainder_sign", "    *r16 = (int16_t)(int32_t)(u - ((uint32_t)hi << 16));\n",
     "    *r16 = (int16_t)(int32_t)(((uint32_t)hi << 16) - u);\n"),
    ("remainder_mode_no_decay", "        float upd = (s.step_size * (m1 / den)) + (s.lrwd * p0);\n        float pn = p0 - upd;\n        m[i] = m1;",
     "        float upd = (s.step_size * (m1 / den));\n        float pn = p0 - upd;\n        m[i] = m1;"),
    ("v32_variance_rounded", "        v[i] = v1;\n        c[i] = f32_to_bf16_rne(y - (pn - p0));\n",
     "        v[i] = bf16_bits_to_f32(f32_to_bf16_rne(v1));\n        c[i] = f32_to_bf16_rne(y - (pn - p0));\n"),
    ("v32_comp_sign", "        c[i] = f32_to_bf16_rne(y - (pn - p0));\n",
     "        c[i] = f32_to_bf16_rne(y + (pn - p0));\n"),
    ("plain_update_sign", "        p[i] = f32_to_bf16_rne(p0 - upd);\n",
     "        p[i] = f32_to_bf16_rne(p0 + upd);\n"),
    ("lr_no_warmup", "    if (k < warmup)\n", "    if (k < 0)\n"),
    ("lr_decay_off_by_one", "        f = (double)(total - k) / span;\n",
     "        f = (double)(total - k - 1) / span;\n"),
    ("clip_scale_ignored_mixed", "float p0 = master[i];\n",
     "float p0 = master[i]; gi = bf16_bits_to_f32(g[i]);\n"),
    ("list_norm_first_tensor_only",
     "        for (int32_t k = 0; k < n_tensors; ++k)\n            oracle_grad_sumsq(",
     "        for (int32_t k = 0; k < 1; ++k)\n            oracle_grad_sumsq("),
    ("list_coef_ignored", "        coef = oracle_clip_coef(acc[0] + acc[1], hp->max_grad_norm, norm_out);",
     "        (void)oracle_clip_coef(acc[0] + acc[1], hp->max_grad_norm, norm_out);"),
    ("list_steps_first_tensor_only",
     "    for (int32_t k = 0; k < n_tensors; ++k) {\n        const oracle_tensor_t* e = &list[k];",
     "    for (int32_t k = 0; k < 1; ++k) {\n        const oracle_tensor_t* e = &list[k];"),
    ("anyprec_fp32_store_rounds", "        ((float*)buf)[i] = x;\n        return x;\n",
     "        x = bf16_bits_to_f32(f32_to_bf16_rne(x));\n        ((float*)buf)[i] = x;\n"
     "        return x;\n"),
    ("anyprec_unrounded_moment_used", "        float ms = store_any(m, m32, i, m1);\n",
     "        float ms = m1; store_any(m, m32, i, m1);\n"),
    ("anyprec_unrounded_variance_used", "        float vs = store_any(v, v32, i, v1);\n",
     "        float vs = v1; store_any(v, v32, i, v1);\n"),
    ("anyprec_comp_sign", "            store_any(c, c32, i, y - (pn - p0));\n",
     "            store_any(c, c32, i, y + (pn - p0));\n"),
    ("anyprec_update_sign", "            float y = load_any(c, c32, i) - upd;\n",
     "            float y = load_any(c, c32, i) + upd;\n"),
    ("anyprec_comp_not_read", "            float y = load_any(c, c32, i) - upd;\n",
     "            float y = 0.0f - upd;\n"),
    ("anyprec_plain_sign", "            p[i] = f32_to_bf16_rne(p0 - upd);\n",
     "            p[i] = f32_to_bf16_rne(p0 + upd);\n"),
    ("anyprec_m_type_ignored", "    const int m32 = (flags & 1) != 0,", "    const int m32 = 0 * (flags & 1),"),
    ("anyprec_v_type_ignored", "v32 = (flags & 2) != 0;", "v32 = 0 * (flags & 2);"),
    ("anyprec_c_type_ignored", "    const int c32 = (flags & 4) != 0,", "    const int c32 = 0 * (flags & 4),"),
    ("anyprec_kahan_ignored", "kahan = (flags & 8) == 0;", "kahan = 0 * (flags & 8);"),
    ("anyprec_no_decay", "        float upd = (s.step_size * (ms / den)) + (s.lrwd * p0);\n\n        if (kahan)",
     "        float upd = (s.step_size * (ms / den));\n\n        if (kahan)"),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutant {name}: text not found in oracle source"
    src = src.replace(old, new)
    cpath = os.path.join(tmp_path, f"{name}.c")
    with open(cpath, "w") as f:
        f.write(src)
    return oracle.load(oracle.compile_source(cpath, os.path.join(tmp_path, f"lib{name}.so")))


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    o = _build_mutant(str(tmp_path), name, old, new)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
            break
    assert caught, f"mutant {name} passed every pin"
