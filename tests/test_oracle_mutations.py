"""Planted mistakes: each case edits a temporary copy of oracle.c in one
plausible way, rebuilds it on the CPU, and checks that at least one of the
oracle's pins now fails.  This shows that the pins constrain every step of
the definition (scale, division, tie rule, stochastic rounding, Philox,
matmul layouts, linear wiring, rescale, bf16 rounding)."""
import os
import shutil
import subprocess
import sys

import pytest

import oracle
from oracle import build as obuild
import test_oracle_linear as L
import test_oracle_philox_mm as PM
import test_oracle_quantize as Q

MUTATIONS = {
    "reciprocal_instead_of_division": ("float v = x / s;", "float v = x * (1.0f / s);"),
    "scale_over_128": ("float s = amax / 127.0f;", "float s = amax / 128.0f;"),
    "ties_away_from_zero": ("return clamp_code(nearbyintf(v));", "return clamp_code(roundf(v));"),
    "sr_comparison_reversed": ("(u < fr) ? f + 1.0f : f", "(u > fr) ? f + 1.0f : f"),
    "philox_key_bumped_before_first_round": ("if (round > 0) {", "if (round >= 0) {"),
    "philox_multiplier_swapped": ("(uint64_t)PHILOX_M0 * (uint64_t)c0", "(uint64_t)PHILOX_M1 * (uint64_t)c0"),
    "b_operand_layout_ignored": ("j->layout == ORC_AxBT ? j->B[jn * j->K + k] : j->B[k * j->N + jn]",
                                 "j->B[jn * j->K + k]"),
    "grad_input_w_grouped_by_rows": ("W, N, K, 1, ORC_STREAM_GI_W", "W, N, K, 0, ORC_STREAM_GI_W"),
    "grad_weight_operands_swapped": ("dY, T, N, 1, ORC_STREAM_GW_DY, X, T, K, 1, ORC_STREAM_GW_X",
                                     "X, T, K, 1, ORC_STREAM_GW_X, dY, T, N, 1, ORC_STREAM_GW_DY"),
    "rescale_drops_column_scale": ("float o = t * sB[j];", "float o = t;"),
    "bf16_truncates": ("bits += 0x7fffu + lsb;", "bits += 0u * lsb;"),
    "bf16_grad_input_untransposed": ("orc_matmul_bf16(dY, W, T, K, N, ORC_AxB, dX, nthreads)",
                                     "orc_matmul_bf16(dY, W, T, K, N, ORC_AxBT, dX, nthreads)"),
    "bf16_pass_rounds_in_fp64_to_bf16_by_truncation": ("j->out[i * j->N + n] = orc_f32_to_bf16_rne((float)s);",
                                                        "j->out[i * j->N + n] = (uint16_t)(orc_f32_to_bf16_rne((float)s) & 0xFFFEu);"),
    "scale_floored_at_epsilon": ("float s = amax / 127.0f;", "float s = fmaxf(amax / 127.0f, 1e-12f);"),
}

PINS = [
    Q.test_golden_4x8_rows_and_columns,
    lambda: Q.test_rne_matches_exact_rational_definition(0),
    lambda: Q.test_rne_invariants((48, 256), 0.01, 20.0, 1),
    Q.test_codes_use_ieee_division_not_reciprocal,
    Q.test_sr_is_unbiased,
    Q.test_sr_exact_values_are_never_moved,
    lambda: PM.test_philox_matches_curand_host_generator(42),
    lambda: PM.test_mm_s32_equals_int64_brute_force(oracle.AxB),
    PM.test_rescale_closed_forms_and_ties,
    lambda: L.test_forward_closed_form(oracle.RNE),
    lambda: L.test_grad_input_closed_form(oracle.RNE),
    lambda: L.test_grad_weight_closed_form(oracle.RNE),
    lambda: L.test_bf16_matmul_matches_exact_rational_product(oracle.AxB),
    L.test_bf16_passes_in_the_linear_layer,
]


def _build_mutant(tmp_path, old, new):
    src = open(os.path.join(os.path.dirname(obuild.__file__), "oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    d = tmp_path / "mutant"
    d.mkdir()
    (d / "oracle.c").write_text(src.replace(old, new))
    shutil.copy(os.path.join(os.path.dirname(obuild.__file__), "oracle.h"), d / "oracle.h")
    lib = d / "liboracle.so"
    subprocess.run(["gcc", *[f for f in obuild.CFLAGS if not f.startswith("-W")],
                    str(d / "oracle.c"), "-o", str(lib), "-lm"], check=True)
    return str(lib)


def run_pins(lib):
    """Child-process body: run every pin against the mutant; exit 3 if one
    fails, 0 if all pass.  A mutant that corrupts memory may crash the child
    instead, which also counts as detected."""
    caught = []
    with oracle.use_library(lib):
        for i, pin in enumerate(PINS):
            try:
                pin()
            except (AssertionError, ValueError):
                caught.append(i)
            except pytest.skip.Exception:
                pass
    print("caught by pins", caught)
    sys.exit(3 if caught else 0)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(name, tmp_path):
    old, new = MUTATIONS[name]
    lib = _build_mutant(tmp_path, old, new)
    here = os.path.dirname(os.path.abspath(__file__))
    code = ("import sys; sys.path[:0] = [%r, %r]; import test_oracle_mutations as m; m.run_pins(%r)"
            % (os.path.dirname(here), here, lib))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"no pin caught the planted mistake {name}:\n{r.stdout}"
