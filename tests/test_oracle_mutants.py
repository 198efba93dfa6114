"""Plant plausible mistakes in a copy of the oracle and require the pins to see them.

Each mutant is the oracle's own C source with one textual change, compiled
into a temporary library on the CPU. A mutant that passes every pin would
mean the pins cannot tell that mistake from the method.
"""

import pytest

import oracle
from tests import oracle_checks as oc

MUTANTS = {
    # frequencies over the whole head width instead of each axis' width
    "freq_full_width": ("pow(theta, -2.0 * (double)j / (double)d_a)",
                        "pow(theta, -2.0 * (double)j / 128.0)"),
    # exponent missing the factor 2
    "freq_no_two": ("pow(theta, -2.0 * (double)j / (double)d_a)",
                    "pow(theta, -1.0 * (double)j / (double)d_a)"),
    # axes read in reverse column order
    "axis_order": ("(double)ids[s * n_axes + a]", "(double)ids[s * n_axes + (n_axes - 1 - a)]"),
    # wrong sign in the rotation
    "rotation_sign": ("y[2 * p] = re * c[p] - im * sn[p];",
                      "y[2 * p] = re * c[p] + im * sn[p];"),
    # rotation by the inverse angle
    "rotation_inverse": ("y[2 * p + 1] = re * sn[p] + im * c[p];",
                         "y[2 * p + 1] = -re * sn[p] + im * c[p];"),
    # split-halves pairing instead of adjacent pairs
    "split_halves": ("double re = x[2 * p], im = x[2 * p + 1];",
                     "double re = x[p], im = x[p + D / 2];"),
    # no 1/sqrt(D) scale
    "no_scale": ("z[j] = acc * scale;", "z[j] = acc;"),
    # softmax not normalised
    "no_normalise": ("double w = z[j] / denom;", "double w = z[j];"),
    # queries left unrotated
    "q_unrotated": ("J->sin_t + i * (D / 2), D, qhat);",
                    "J->sin_t + i * (D / 2), D, qhat); for (int c = 0; c < D; ++c) "
                    "qhat[c] = J->q[qoff + c];"),
    # keys rotated with the query's position
    "k_wrong_position": ("J->cos_t + j * (D / 2),\n                          J->sin_t + j * (D / 2)",
                         "J->cos_t + 0 * (D / 2),\n                          J->sin_t + 0 * (D / 2)"),
    # values read from the key tensor
    "v_from_k": ("const double *vj = J->v +", "const double *vj = J->k +"),
    # QK norm: eps added outside the square root
    "norm_eps_outside": ("1.0 / sqrt(ss / (double)D + eps)", "1.0 / (sqrt(ss / (double)D) + eps)"),
    # QK norm: sum of squares instead of their mean
    "norm_sum_not_mean": ("sqrt(ss / (double)D + eps)", "sqrt(ss + eps)"),
    # QK norm: learned weight ignored
    "norm_no_weight": ("y[c] = x[c] * r * w[c];", "y[c] = x[c] * r;"),
    # QK norm: text and image key weights swapped
    "norm_segments_swapped": ("j < J->S_txt ? J->kw_txt : J->kw_img",
                              "j < J->S_txt ? J->kw_img : J->kw_txt"),
    # QK norm: keys normalised with the query weights
    "norm_k_with_q_weights": ("j < J->S_txt ? J->kw_txt : J->kw_img",
                              "j < J->S_txt ? J->qw_txt : J->qw_img"),
    # QK norm: segment boundary off by one for the queries
    "norm_segment_off_by_one": ("i < J->S_txt ? J->qw_txt", "i <= J->S_txt ? J->qw_txt"),
    # KV modes: no 1/sqrt(D) scale
    "range_no_scale": ("z[j] = scale * acc;", "z[j] = acc;"),
    # KV modes: softmax not normalised
    "range_no_normalise": ("const double wj = z[j] / denom;", "const double wj = z[j];"),
    # extract: reference queries attend to every key
    "extract_ref_sees_all": ("is_ref ? S_txt : 0, is_ref ? S_txt + S_ref : S",
                             "0, S"),
    # extract: text and image queries restricted to the reference keys too
    "extract_all_restricted": ("is_ref ? S_txt : 0, is_ref ? S_txt + S_ref : S",
                               "S_txt, S_txt + S_ref"),
    # extract: the cache holds the unrotated keys
    "extract_cache_unrotated": ("cache_k[coff + c] = khat[(S_txt + r) * D + c];",
                                "cache_k[coff + c] = k[(((int64_t)b * S + S_txt + r) * H + h) * D + c];"),
    # cached: the cached keys rotated again by the query-side table
    "cached_rerotated": ("for (int c = 0; c < D; ++c) khat[j * D + c] = cache_k[coff + c];",
                         "oracle_rope_apply_vec(cache_k + coff, cos_t, sin_t, D, khat + j * D);"),
    # cached: image keys read from the wrong token (offset by the cache length)
    "cached_img_offset": ("const int64_t t = j < S_txt ? j : j - S_ref;",
                          "const int64_t t = j < S_txt ? j : (j - S_ref + 1) % S;"),
    # off-by-one in the key loop
    "skip_last_key": ("for (int64_t j = 0; j < S; ++j) {\n      double acc",
                      "for (int64_t j = 0; j < S - 1; ++j) {\n      double acc"),
    "kvnorm_k_with_q_weights": ("oracle_rms_norm_vec(k + off, t < S_txt ? kw_txt : kw_img, D, eps, *kn + off);",
                                "oracle_rms_norm_vec(k + off, t < S_txt ? qw_txt : qw_img, D, eps, *kn + off);"),
    "kvnorm_refs_as_text": ("oracle_rms_norm_vec(q + off, t < S_txt ? qw_txt : qw_img, D, eps, *qn + off);",
                            "oracle_rms_norm_vec(q + off, t < S_txt + 4 ? qw_txt : qw_img, D, eps, *qn + off);"),
    "proj_gate_linear_swapped": ("proj_dot(xi, w, dim, n_out, 3 * inner + j);",
                                 "proj_dot(xi, w, dim, n_out, 3 * inner + mlp + j);"),
    "proj_no_sigmoid": ("act[r * mlp + j] = g / (1.0 + exp(-g)) * u;",
                        "act[r * mlp + j] = g * u;"),
    "proj_sigmoid_sign": ("act[r * mlp + j] = g / (1.0 + exp(-g)) * u;",
                          "act[r * mlp + j] = g / (1.0 + exp(g)) * u;"),
    "proj_k_from_q": ("proj_dot(xi, w, dim, n_out, inner + c);",
                      "proj_dot(xi, w, dim, n_out, c);"),
    "proj_v_from_k": ("proj_dot(xi, w, dim, n_out, 2 * inner + c);",
                      "proj_dot(xi, w, dim, n_out, inner + c);"),
    "proj_weight_transposed": ("acc += wn[c] * x[c];", "acc += w[(int64_t)c * n_out + n] * x[c];"),
    "proj_last_channel_skipped": ("for (int c = 0; c < dim; ++c) acc += wn[c]",
                                  "for (int c = 0; c < dim - 1; ++c) acc += wn[c]"),
}


def _run_checks(orc):
    failed = []
    for check in oc.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
        except ImportError:
            pass
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    pytest.importorskip("mpmath")
    src = open(oracle.SOURCE).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    mpath = tmp_path / f"mutant_{name}.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mpath), str(tmp_path / f"libmutant_{name}.so"))
    failed = _run_checks(oracle.Oracle(lib))
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_source_passes(tmp_path):
    pytest.importorskip("mpmath")
    lib = oracle.compile_source(oracle.SOURCE, str(tmp_path / "libclean.so"))
    assert _run_checks(oracle.Oracle(lib)) == []
