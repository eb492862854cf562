"""The oracle's pins catch plausible mistakes -- CPU only.

Each case plants one mistake (a flipped tie rule, a wrong comparison, a
dropped factor, a transposed index, a wrong constant, a wrong rounding mode
or shared random stream in the MLP composition) in a *copy* of the oracle's
source -- never in the oracle itself -- builds the copy as a
separate package in a temporary directory and runs the pins that should
notice it: at least one must fail.  The unmutated copy passes the same pins
(the control), so a failure means the pin saw the mistake, not that the
copy is broken.  (Saturating E4M3 only from 480 is no such case: the
encoder's final clamp to 0x7E gives the same codes.)
"""
import importlib.util
import itertools
import os
import shutil
import sys

import pytest

import test_oracle_formats as formats
import test_oracle_gemm as gemm
import test_oracle_mlp as mlp
import test_oracle_mx as mx
import test_oracle_philox as philox
import test_oracle_quantize as quantize
import test_oracle_rht as rht

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_COPIES = itertools.count()

# name -> (substitutions (old, new) in nvfp4_oracle.c, or (file, old, new),
#          pins that must catch it)
MUTANTS = {
    "E2M1 ties away from zero": (
        [("else pick = ((lo & 1) == 0) ? lo : hi;", "else pick = hi;")],
        [formats.test_e2m1_ties_to_even]),
    "SR rounds up on r == threshold": (
        [("int up = (double)rbits < thr;", "int up = (double)rbits <= thr;")],
        [formats.test_e2m1_sr_rule]),
    "E4M3 subnormal range ends at 2^-7": (
        [("if (a < ldexp(1.0, -6)) {", "if (a < ldexp(1.0, -7)) {")],
        [formats.test_e4m3_saturation_and_subnormals]),
    "E4M3 subnormal step 2^-10": (
        [("double n = rint(a * 512.0);", "double n = rint(a * 1024.0);")],
        [formats.test_e4m3_saturation_and_subnormals]),
    "RHT scaled by 1/2 instead of 1/4": (
        [("for (int i = 0; i < 16; ++i) v[i] = v[i] * 0.25f;",
          "for (int i = 0; i < 16; ++i) v[i] = v[i] * 0.5f;")],
        [rht.test_butterfly_builds_the_sylvester_matrix,
         rht.test_rht_cancels_in_the_wgrad_product]),
    "RHT butterfly difference reversed": (
        [("v[i + h] = a - b;", "v[i + h] = b - a;")],
        [rht.test_butterfly_builds_the_sylvester_matrix]),
    "Philox Weyl constant off by one": (
        [("k1 += 0xBB67AE85u;", "k1 += 0xBB67AE86u;")],
        [philox.test_philox_matches_triton_interpreter]),
    "SR word taken from the neighbouring lane": (
        [("return out[idx & 3];", "return out[(idx + 1) & 3];")],
        [philox.test_sr_word_layout]),
    "scale layout with row quarter and column swapped": (
        [("return atom * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4);",
          "return atom * 512 + (r % 32) * 16 + (c % 4) * 4 + ((r / 32) % 4);")],
        [quantize.test_swizzle_matches_reshape_formulation]),
    "nibbles packed high first": (
        [("if ((j & 1) == 0) row[j / 2]", "if ((j & 1) == 1) row[j / 2]")],
        [lambda o: quantize.test_row_quantize_brute_force(o, "bf16", (32, 64))]),
    "zero tensor gets s_enc = 0": (
        [("if (amax == 0.0f) return 1.0f;", "if (amax == 0.0f) return 0.0f;")],
        [quantize.test_zero_tensor_and_amax_given]),
    "block scale without the division by 6": (
        [("float t = (a_b / 6.0f) * s_enc;", "float t = a_b * s_enc;")],
        [lambda o: quantize.test_row_quantize_brute_force(o, "bf16", (32, 64))]),
    "GEMM reads B transposed": (
        [("acc += a[m * K + k] * b[n * K + k];", "acc += a[m * K + k] * b[k * N + n];")],
        [lambda o: gemm.test_gemm_reduces_to_textbook_gemm(o, 8, 12, 16)]),
    "16x16 transposed scales taken from the wrong tile": (
        [("out->scales_t[(tc * 16 + j) * (orows / 16) + tr] = sc;",
          "out->scales_t[(tc * 16 + j) * (orows / 16) + (orows / 16 - 1 - tr)] = sc;")],
        [quantize.test_16x16_one_scale_per_tile_and_transpose_invariant]),
    "SR window ignores its index base": (
        [("orc_sr_word(seed, offset, sr_index_base + (uint64_t)(r * ocols + c))",
          "orc_sr_word(seed, offset, (uint64_t)(r * ocols + c))")],
        [quantize.test_sr_window_equals_slab_of_whole]),
    "BF16 rounding by truncation": (
        [("double q = rint(ldexp(a, -lsb_exp));", "double q = floor(ldexp(a, -lsb_exp));")],
        [formats.test_bf16_from_double_is_nearest_even]),
    "SwiGLU with sigmoid(-g)": (
        [("static double sigmoid_d(double g) { return 1.0 / (1.0 + exp(-g)); }",
          "static double sigmoid_d(double g) { return 1.0 / (1.0 + exp(g)); }")],
        [mlp.test_swiglu_matches_autograd]),
    # the MX comparison formats
    "E8M0 shared exponent offset 1 for E2M1": (
        [("const int emax = fmt == ORC_MXFP8 ? 8 : 2;", "const int emax = fmt == ORC_MXFP8 ? 8 : 1;")],
        [lambda o: mx.test_e8m0_scale_closed_forms(o, mx.MXFP4)]),
    "MX elements scaled by twice the block scale": (
        [("const float y = (float)ldexp((double)v[i], -((int)sb - 127));",
          "const float y = (float)ldexp((double)v[i], -((int)sb - 126));")],
        [lambda o: mx.test_elements_are_the_nearest_code(o, mx.MXFP4)]),
    "MX column mode reads along rows": (
        [("const int64_t idx = mode == ORC_MX_ROW ? r * ld + c : c * ld + r;",
          "const int64_t idx = mode == ORC_MX_ROW ? r * ld + c : r * ld + c;")],
        [lambda o: mx.test_column_mode_is_row_mode_of_transpose(o, mx.MXFP4)]),
    "MX all-zero block drops the sign of zero": (
        [("code = fmt == ORC_MXFP4 ? 0x8 : 0x80;  /* -0 in an all-zero block */", "code = 0;")],
        [mx.test_zero_and_nonfinite_blocks]),
    # the MLP composition (the recipe's per-operand choices)
    "dG rounded to nearest instead of stochastically": (
        [("mlp.py", 'qdG = quantize(dG, ROW_1X16, SR, seed=seed, offset=off["dg_row"])',
          'qdG = quantize(dG, ROW_1X16, 0, seed=seed, offset=off["dg_row"])')],
        [lambda o: mlp.test_mlp_gradient_operands_are_stochastically_rounded(
            o, mlp.make_mlp_run(o))]),
    "dU's row operand reuses dG's SR offset": (
        [("mlp.py", '"du_row": b + 4', '"du_row": b + 2')],
        [lambda o: mlp.test_mlp_sr_operands_draw_independent_words(o, mlp.make_mlp_run(o))]),
    "H's WGRAD operand without the RHT": (
        [("mlp.py", "qHc = quantize(H, COL_1X16, rf, seed=seed)",
          "qHc = quantize(H, COL_1X16, 0, seed=seed)")],
        [lambda o: mlp.test_mlp_wgrad_operands_carry_the_rht(o, mlp.make_mlp_run(o))]),
    "dX without the up projection's term": (
        [("mlp.py", "dX = bf16_round_f64(gemm_fp64(qdG, transposed_view(saved[\"qWg\"])) +\n"
                    "                        gemm_fp64(qdU, transposed_view(saved[\"qWu\"])))",
          "dX = bf16_round_f64(gemm_fp64(qdG, transposed_view(saved[\"qWg\"])))")],
        [lambda o: mlp.test_nvfp4_mlp_tracks_fp64_mlp(o, True)]),
    "SGD with the rate's sign flipped": (
        [("mlp.py", "W_new = np.subtract(", "W_new = np.add(")],
        [mlp.test_sgd_step_exact_on_representable_values]),
}


def _copy_oracle(dst, subs):
    """The oracle package copied to dst with `subs` applied to its C source,
    imported under a name of its own (it builds its own library in dst)."""
    src = os.path.join(ROOT, "oracle")
    os.makedirs(dst)
    for f in ("__init__.py", "mlp.py", "nvfp4_oracle.c", "nvfp4_oracle.h"):
        shutil.copy(os.path.join(src, f), os.path.join(dst, f))
    for sub in subs:
        fname, old, new = sub if len(sub) == 3 else ("nvfp4_oracle.c", *sub)
        path = os.path.join(dst, fname)
        code = open(path).read()
        assert code.count(old) == 1, f"mutation site not unique: {old!r}"
        open(path, "w").write(code.replace(old, new))
    name = f"oracle_copy_{next(_COPIES)}"  # a fresh package (and mlp submodule) per copy
    spec = importlib.util.spec_from_file_location(
        name, os.path.join(dst, "__init__.py"), submodule_search_locations=[dst])
    mod = importlib.util.module_from_spec(spec)
    sys.modules[name] = mod
    spec.loader.exec_module(mod)
    mod.build()
    return mod


def _pins_fail(orc, pins):
    failed = []
    for pin in pins:
        try:
            pin(orc)
        except (AssertionError, ValueError) as e:
            failed.append((pin, e))
    return failed


def test_unmutated_copy_passes_every_pin(tmp_path):
    orc = _copy_oracle(str(tmp_path / "control"), [])
    pins = [p for _, ps in MUTANTS.values() for p in ps]
    assert not _pins_fail(orc, pins)


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    subs, pins = MUTANTS[name]
    orc = _copy_oracle(str(tmp_path / "mutant"), subs)
    assert _pins_fail(orc, pins), f"no pin noticed: {name}"
