"""Pin strength: plant a plausible mistake in a copy of the oracle's C source
(a dropped term, a wrong beta, a flipped sign or comparison, a wrong index),
build it, and check that at least one pin of tests/test_oracle_pins.py fails.
Every mistake is planted in the oracle, on the CPU."""
import pytest

import oracle
import test_oracle_pins as pins

# (name, original text, planted text, pins expected to catch it)
MUTANTS = [
    ("map half-step offset dropped", "((double)f + 0.5)", "((double)f + 0.0)",
     [(pins.test_qmap_matches_byte_structure_enumeration, (True,))]),
    ("map exponent off by one", "pow(10.0, -(double)k)", "pow(10.0, -(double)k - 1.0)",
     [(pins.test_qmap_closed_form_values, ())]),
    ("midpoint scale", "(q[i] + q[i + 1]) * 0.5f", "(q[i] + q[i + 1]) * 0.45f",
     [(pins.test_code_is_nearest_level_brute_force, (pins.S,))]),
    ("tie goes up", "if (mid[i] < xn) c += 1;", "if (mid[i] <= xn) c += 1;",
     [(pins.test_code_tie_goes_to_lower_level_and_exact_levels_map_to_themselves, ())]),
    ("no reciprocal of absmax", "return absmax > 0.0f ? 1.0f / absmax : 0.0f;",
     "return absmax > 0.0f ? absmax : 0.0f;",
     [(pins.test_quantize_round_trips_every_level, (256, 5))]),
    ("absmax of block 0 for every element", "return s->q[((const uint8_t*)s->base)[i]] * s->absmax[i / B];",
     "return s->q[((const uint8_t*)s->base)[i]] * s->absmax[0];",
     [(pins.test_8bit_step_tracks_32bit, ("adam", "f32"))]),
    ("Adam m with beta2", "float m = fmaf(sc->b1, s_old[0], sc->omb1 * g);\n      float v",
     "float m = fmaf(sc->b2, s_old[0], sc->omb2 * g);\n      float v",
     [(pins.test_32bit_step_matches_torch_optim, ("adam", 0.0, 1.0))]),
    ("Adam v not squared", "float v = fmaf(sc->b2, s_old[1], sc->omb2 * (g * g));",
     "float v = fmaf(sc->b2, s_old[1], sc->omb2 * fabsf(g));",
     [(pins.test_32bit_step_matches_torch_optim, ("adam", 0.0, 1.0))]),
    ("Adam eps without bias correction", "sc->eps_hat = (float)(eps * sqrt(bc2));\n      sc->unorm_c = sqrt(bc2) / bc1;",
     "sc->eps_hat = (float)(eps);\n      sc->unorm_c = sqrt(bc2) / bc1;",
     [(pins.test_32bit_step_matches_torch_optim, ("adam", 0.0, 1.0))]),
    ("Adam step without sqrt(bc2)", "sc->step_size = (float)(lr * sqrt(bc2) / bc1);",
     "sc->step_size = (float)(lr / bc1);",
     [(pins.test_32bit_step_matches_torch_optim, ("adam", 0.0, 1.0))]),
    ("coupled decay sign", "g = fmaf(wd, p, g);", "g = fmaf(-wd, p, g);",
     [(pins.test_32bit_step_matches_torch_optim, ("adam", 1e-2, 1.0))]),
    ("decoupled decay dropped", "if (decoupled(hp->optim) && wd != 0.0f) p = p * sc->decay;",
     "if (0) p = p * sc->decay;",
     [(pins.test_32bit_step_matches_torch_optim, ("adamw", 1e-2, 1.0))]),
    ("gnorm_scale ignored", "float g = g_raw * hp->gnorm_scale;", "float g = g_raw;",
     [(pins.test_32bit_step_matches_torch_optim, ("momentum", 0.0, 0.5))]),
    ("momentum dampened", "float m = fmaf(sc->b1, s_old[0], g);",
     "float m = fmaf(sc->b1, s_old[0], sc->omb1 * g);",
     [(pins.test_32bit_step_matches_torch_optim, ("momentum", 0.0, 1.0))]),
    ("RMSprop without (1-alpha)", "float v = fmaf(sc->b1, s_old[0], sc->omb1 * (g * g));",
     "float v = fmaf(sc->b1, s_old[0], (g * g));",
     [(pins.test_32bit_step_matches_torch_optim, ("rmsprop", 0.0, 1.0))]),
    ("Adagrad state not squared", "float v = fmaf(g, g, s_old[0]);", "float v = s_old[0] + fabsf(g);",
     [(pins.test_32bit_step_matches_torch_optim, ("adagrad", 0.0, 1.0))]),
    ("Lion c with beta2", "float c = fmaf(sc->b1, s_old[0], sc->omb1 * g);",
     "float c = fmaf(sc->b2, s_old[0], sc->omb2 * g);",
     [(pins.test_lion_worked_example, ())]),
    ("Lion sign flipped", "u = c > 0.0f ? 1.0f : (c < 0.0f ? -1.0f : 0.0f);",
     "u = c > 0.0f ? -1.0f : (c < 0.0f ? 1.0f : 0.0f);",
     [(pins.test_lion_worked_example, ())]),
    ("Lion momentum with beta1", "r.s[0] = fmaf(sc->b2, s_old[0], sc->omb2 * g);",
     "r.s[0] = fmaf(sc->b1, s_old[0], sc->omb1 * g);",
     [(pins.test_lion_constant_gradient_closed_form, ())]),
    ("AdEMAMix m2 with beta1", "float m2 = fmaf(sc->b3t, s_old[1], sc->omb3t * g);",
     "float m2 = fmaf(sc->b1, s_old[1], sc->omb1 * g);",
     [(pins.test_ademamix_constant_gradient_closed_form, ())]),
    ("AdEMAMix alpha on m1", "sc->alpha_t * m2", "sc->alpha_t * m1",
     [(pins.test_ademamix_constant_gradient_closed_form, ())]),
    ("AdEMAMix m1 not bias-corrected", "fmaf(m1, sc->inv_bc1, sc->alpha_t * m2)",
     "(m1 + sc->alpha_t * m2)",
     [(pins.test_ademamix_alpha_zero_is_adamw, ())]),
    ("AdEMAMix nu with beta1", "float nu = fmaf(sc->b2, s_old[2], sc->omb2 * (g * g));",
     "float nu = fmaf(sc->b1, s_old[2], sc->omb1 * (g * g));",
     [(pins.test_ademamix_alpha_zero_is_adamw, ())]),
    ("alpha warm-up inverted", "at = ramp < a ? ramp : a;", "at = ramp > a ? ramp : a;",
     [(pins.test_ademamix_schedules_endpoints_and_monotone, ())]),
    ("beta3 warm-up clamps the wrong way", "b3t = s < b3 ? s : b3;", "b3t = s > b3 ? s : b3;",
     [(pins.test_ademamix_schedules_endpoints_and_monotone, ())]),
    ("beta3 warm-up interpolates the wrong ends", "((1.0 - r) * lb3 + r * lb1)",
     "((1.0 - r) * lb1 + r * lb3)",
     [(pins.test_ademamix_schedules_endpoints_and_monotone, ())]),
    ("skip test after decay", "r.skipped = hp->skip_zeros && g_raw == 0.0f;",
     "r.skipped = hp->skip_zeros && g_raw + hp->weight_decay * p == 0.0f;",
     [(pins.test_skip_zeros_identities, ("adam", 8, "f32"))]),
    ("fully skipped block requantized", "if (!any_update) continue;", "if (0) continue;",
     [(pins.test_skip_zeros_identities, ("momentum", 8, "f32"))]),
    ("requantization absmax without |.|", "float a = fabsf(x[i]);", "float a = x[i];",
     [(pins.test_8bit_step_tracks_32bit, ("momentum", "f32"))]),
    ("requantization absmax skips a NaN", "    if (isnan(a)) return a;\n", "",
     [(pins.test_step_nan_state_makes_its_block_absmax_nan, ())]),
    ("quantization absmax skips a NaN", "      if (isnan(a)) { amax = a; break; }\n", "",
     [(pins.test_quantize_nan_makes_its_block_absmax_nan, ())]),
    ("AdEMAMix m2 aliases m1", "out[1].base = (char*)s1 + n * esz;", "out[1].base = (char*)s1;",
     [(pins.test_8bit_step_tracks_32bit, ("ademamix", "f32"))]),
    ("update norm not squared",
     "usum += (double)r.u * (double)r.u;\n    psum += (double)pv * (double)pv;\n  }\n  double unorm = sc.unorm_c",
     "usum += fabs((double)r.u);\n    psum += (double)pv * (double)pv;\n  }\n  double unorm = sc.unorm_c",
     [(pins.test_max_unorm_norms_match_numpy, ())]),
    ("parameter norm taken after the step",
     "psum += (double)pv * (double)pv;\n  }\n  double unorm = sc.unorm_c",
     "psum += (double)r.p * (double)r.p;\n  }\n  double unorm = sc.unorm_c",
     [(pins.test_max_unorm_norms_match_numpy, ())]),
    ("clip applied to states too", "if (decoupled(hp->optim) && wd != 0.0f) p = p * sc->decay;\n  r.p = fmaf(-step_eff, u, p);",
     "if (decoupled(hp->optim) && wd != 0.0f) p = p * sc->decay;\n  r.p = fmaf(-step_eff, u, p);\n  for (int j = 0; j < 3; ++j) r.s[j] *= step_eff / sc->step_size;",
     [(pins.test_max_unorm_invariants, ("momentum",))]),
    ("parameter moves up the update", "r.p = fmaf(-step_eff, u, p);", "r.p = fmaf(step_eff, u, p);",
     [(pins.test_32bit_step_matches_torch_optim, ("adam", 0.0, 1.0))]),
    ("per-block clip over the whole tensor",
     "block_unorm_scale(hp, &sc, p, g, st, ns, 8, dtype, B, lo, hi)",
     "block_unorm_scale(hp, &sc, p, g, st, ns, 8, dtype, B, 0, n)",
     [(pins.test_max_unorm_per_block_invariants, ("momentum", 8))]),
    ("per-block parameter norm after the step", "    psum += (double)pv * (double)pv;\n  }\n  double unorm = sc->unorm_c",
     "    psum += (double)r.p * (double)r.p;\n  }\n  double unorm = sc->unorm_c",
     [(pins.test_max_unorm_per_block_invariants, ("adam", 8))]),
    ("parameter norm without squares", "    psum += v * v;\n  }\n  return psum;",
     "    psum += fabs(v);\n  }\n  return psum;",
     [(pins.test_param_sumsq_closed_forms, ("f32",))]),
    ("parameter norm drops the last element",
     "for (int64_t i = 0; i < n; ++i) {\n    const double v = (double)load_elem(p, dtype, i);",
     "for (int64_t i = 0; i + 1 < n; ++i) {\n    const double v = (double)load_elem(p, dtype, i);",
     [(pins.test_param_sumsq_closed_forms, ("bf16",))]),
    ("parameter norm squares in binary32",
     "const double v = (double)load_elem(p, dtype, i);\n    psum += v * v;",
     "const float v = load_elem(p, dtype, i);\n    psum += (double)(v * v);",
     [(pins.test_param_sumsq_matches_an_exactly_rounded_sum, ())]),
    ("bf16 rounds half up", "u += 0x7fffu + kept_lsb;", "u += 0x8000u;",
     [(pins.test_bf16_rounding_matches_torch, ())]),
    ("f16 subnormals truncated", "nearbyintf(fa * 16777216.0f)", "floorf(fa * 16777216.0f)",
     [(pins.test_f16_rounding_matches_numpy, ())]),
]


@pytest.mark.parametrize("name,orig,planted,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, orig, planted, checks):
    src = oracle.source_text()
    assert src.count(orig) == 1, f"mutation site for '{name}' not unique"
    lib = oracle.compile_variant(src.replace(orig, planted), str(tmp_path / "mutant.so"))
    caught = []
    with oracle.using_library(lib):
        for fn, args in checks:
            try:
                fn(*args)
            except (AssertionError, FloatingPointError, ValueError) as e:
                caught.append(f"{fn.__name__}: {type(e).__name__}")
    assert caught, f"planted mistake '{name}' passed every pin"


def test_unmutated_source_passes_the_same_pins(tmp_path):
    lib = oracle.compile_variant(oracle.source_text(), str(tmp_path / "same.so"))
    with oracle.using_library(lib):
        for _, _, _, checks in MUTANTS:
            for fn, args in checks:
                fn(*args)
