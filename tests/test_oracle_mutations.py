"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each.

Every mutation edits one spot of oracle.c (a dropped term, a wrong sign or
index, a swapped operand), is compiled on the CPU into a temporary library,
and must make at least one of the pin checks fail: the pages' worked
examples, the Resize pins, the dense brute force, the torch cross-checks,
the DeformConv special cases or the Resize operator's own pins.  A mutation that no pin notices would mean the
oracle could carry that mistake silently.  All mutations keep memory access
in bounds.
"""
import os

import pytest

import oracle
import test_oracle_pages as pages
import test_oracle_pins as pins
import test_oracle_resize as resize_pins
from conftest import fixture_names

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()

MUTATIONS = {
    "keys_tap_order_mirrored": ("w[k] = keys(t + 1.0 - (double)k, a);",
                                "w[k] = keys(t - 1.0 + (double)k, a);"),
    "cubic_first_tap_shifted": ("int64_t j = i0 - 1 + k;", "int64_t j = i0 + k;"),
    "keys_inner_sign": ("- (a + 3.0) * s * s + 1.0", "+ (a + 3.0) * s * s + 1.0"),
    "keys_outer_constant": ("+ 8.0 * a * s - 4.0 * a", "+ 8.0 * a * s + 4.0 * a"),
    "unnormalize_ac0_missing_half_pixel": ("((g + 1.0) * (double)n - 1.0) / 2.0",
                                           "((g + 1.0) * (double)n) / 2.0"),
    "unnormalize_ac1_uses_n": ("(g + 1.0) / 2.0 * (double)(n - 1)", "(g + 1.0) / 2.0 * (double)n"),
    "reflection_ac0_at_centres": ("return reflect(x, -0.5, (double)n - 0.5);",
                                  "return reflect(x, 0.0, (double)(n - 1));"),
    "reflection_no_mirror_half": ("if (m > span) m = 2.0 * span - m;", "if (m > span) m = m - span;"),
    "nearest_rounds_half_up": ("idx[0] = to_index(nearbyint(x));", "idx[0] = to_index(floor(x + 0.5));"),
    "linear_weights_swapped": ("idx[0] = i0;     w[0] = 1.0 - t;", "idx[0] = i0;     w[0] = t;"),
    "border_clip_to_n": ("x = clip(x, 0.0, (double)(n - 1));\n        } else if",
                         "x = clip(x, -0.5, (double)(n - 1));\n        } else if"),
    "grid_vector_order_reversed": ("axis_taps(g[r - 1 - d]", "axis_taps(g[d]"),
    "base_coord_ac0_left_edge": ("return (2.0 * (double)i + 1.0) / (double)n - 1.0;",
                                 "return 2.0 * (double)i / (double)n - 1.0;"),
    "theta_transposed": ("theta_n[row * (r + 1) + k]", "theta_n[k * r + row]"),
    "deform_offsets_swapped": ("* 2 * K + 2 * k) * plane + pix];\n                double dx",
                               "* 2 * K + 2 * k + 1) * plane + pix];\n                double dx"),
    "deform_mask_dropped": ("double v = bilinear_zero(X_nc, H, Wd, y, x) * m;",
                            "double v = bilinear_zero(X_nc, H, Wd, y, x);"),
    "deform_stride_dropped": ("(double)(oh * at->strides[0] - at->pads[0]",
                              "(double)(oh - at->pads[0]"),
    "deform_pad_sign": ("(double)(ow * at->strides[1] - at->pads[1]",
                        "(double)(ow * at->strides[1] + at->pads[1]"),
    "deform_group_offset_ignored": ("int64_t c = g * Cg + ci;", "int64_t c = ci;"),
    "deform_dilation_dropped": ("+ kw * at->dilations[1]) + dx", "+ kw) + dx"),
    "resize_nearest_prefer_floor_rounds_up": ("default: return ceil(x - 0.5);",
                                              "default: return floor(x + 0.5);"),
    "resize_half_pixel_no_shift": ("default: /* half_pixel */\n            return (xr + 0.5) / scale - 0.5;",
                                   "default: /* half_pixel */\n            return xr / scale;"),
    "resize_align_corners_floored_length": (
        "xr * (double)(n_in - 1) / (length_resized - 1.0)",
        "xr * (double)(n_in - 1) / ((double)n_out - 1.0)"),
    "resize_antialias_unnormalised": ("if (s < 1.0) {\n            for (int k = 0; k < cnt; ++k) w[k] /= sum;",
                                      "if (s < 0.0) {\n            for (int k = 0; k < cnt; ++k) w[k] /= sum;"),
    "resize_antialias_unstretched": ("const double d = ((double)k - t) * s;",
                                     "const double d = ((double)k - t);"),
    "resize_exclude_outside_no_renorm": ("if (sum != 0.0)\n            for (int k = 0; k < cnt; ++k) w[k] /= sum;",
                                         "if (sum != sum)\n            for (int k = 0; k < cnt; ++k) w[k] /= sum;"),
    "resize_crop_never_extrapolates": ("if (coord == RS_TF_CROP_AND_RESIZE && (x < 0.0 || x > (double)(n_in - 1))) return -1;",
                                       "if (coord == RS_TF_CROP_AND_RESIZE && (x < -1e300)) return -1;"),
    "resize_keep_policy_inverted": ("(keep_policy == RS_NOT_LARGER ? r < common : r > common)",
                                    "(keep_policy == RS_NOT_LARGER ? r > common : r < common)"),
    "resize_round_int_down": ("floor(common * (double)in_shape[d] + 0.5)",
                              "floor(common * (double)in_shape[d])"),
    "resize_roi_axes_reversed": ("roi_start[ax[i]] = roi[i];", "roi_start[ax[i]] = roi[na - 1 - i];"),
    "resize_scaled_extent_rounded_up": ("out_shape[d] = (int64_t)floor(len);",
                                        "out_shape[d] = (int64_t)ceil(len);"),
    "resize_pytorch_half_pixel_single_not_zero": (
        "return n_out > 1 ? (xr + 0.5) / scale - 0.5 : 0.0;", "return (xr + 0.5) / scale - 0.5;"),
    "resize_cubic_antialias_linear_reach": ("const double reach = mode == OR_LINEAR ? 1.0 : 2.0;",
                                            "const double reach = mode == OR_LINEAR ? 1.0 : 1.0;"),
    "resize_nearest_ceil_as_floor": ("case RS_CEIL: return ceil(x);", "case RS_CEIL: return floor(x);"),
}


def _run_pins():
    """Run the pin checks; return the names of those that failed."""
    failed = []

    def attempt(label, fn, *args):
        try:
            fn(oracle, *args)
        except AssertionError:
            failed.append(label)

    for n in fixture_names("affinegrid__"):
        attempt(n, pages.test_affine_grid_page_example, n)
    for n in fixture_names("gridsample__"):
        attempt(n, pages.test_grid_sample_page_example, n)
    for n in fixture_names("deformconv__"):
        attempt(n, pages.test_deform_conv_page_example, n)
    for n in pages.resize_via_grid_sample_names():
        attempt(n, pages.test_resize_examples_through_grid_sample, n)
    for case in [(2, m, p, ac) for m in ("linear", "nearest", "cubic")
                 for p in ("zeros", "border", "reflection") for ac in (0, 1)]:
        attempt(f"brute{case}", pins.test_tap_oracle_matches_dense_brute_force, *case)
    for case in pins.DEFORM_CASES:
        attempt(f"conv{case}", pins.test_deform_conv_with_zero_offsets_is_conv2d, case)
        attempt(f"bilinear{case}", pins.test_deform_conv_is_a_contraction_of_bilinear_samples, case)
    for r, ac in ((2, 0), (2, 1), (3, 0), (3, 1)):
        attempt(f"affine_torch{r}{ac}", pins.test_affine_grid_matches_torch_cpu_fp64, r, ac)
    for n in fixture_names("resize__"):
        attempt(f"resize_page{n}", resize_pins.test_resize_page_example, n)
    attempt("resize_repeat", resize_pins.test_nearest_double_asymmetric_is_repeat)
    attempt("resize_1331", resize_pins.test_antialias_linear_half_is_1331_filter)
    attempt("resize_crop", resize_pins.test_crop_and_resize_whole_roi_is_identity)
    attempt("resize_extent", resize_pins.test_scale_output_extent_is_floored)
    return failed


def test_unmutated_oracle_passes_every_pin():
    assert _run_pins() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTATIONS[name]
    assert SRC.count(old) == 1, f"mutation anchor not unique: {name}"
    path = oracle.build_variant(SRC.replace(old, new), str(tmp_path / f"mut_{name}.so"))
    with oracle.use_library(path):
        failed = _run_pins()
    assert failed, f"no pin caught the planted mistake {name}"
