"""Planted mistakes in copies of the oracle must each fail at least one pin.

Every mutant below is a plausible slip (a dropped term, a wrong sign or index,
a transposed operand, an off-by-one in the shard plan, halo or crop).  The
mutant is compiled from a modified copy of oracle.c in a temporary directory;
the oracle itself is never changed.  Mutations keep every memory access in
bounds, so a mutant can only compute wrong numbers, never crash the process.
"""
import os

import pytest

import oracle
import oracle_pins as P

# (name, function whose body is edited, old text, new text)
MUTANTS = [
    ("fwd_drops_bias", "int or_conv2d_fwd(", "double acc = b ? (double)b[co] : 0.0;", "double acc = 0.0;"),
    ("fwd_tap_off_by_one", "int or_conv2d_fwd(", "const int c = j * s - p + v;", "const int c = j * s - p + v + (v == 0);"),
    ("fwd_weight_transposed", "int or_conv2d_fwd(", "W4(w, Cgi, d->kh, d->kw, co, cl, u, v)", "W4(w, Cgi, d->kh, d->kw, co, cl, v, u)"),
    ("bwd_input_flipped_row", "int or_conv2d_bwd_input(", "const int h = i * s - p + u;", "const int h = i * s - p + (d->kh - 1 - u);"),
    ("bwd_weight_first_image_only", "int or_conv2d_bwd_weight(", "for (int n = 0; n < d->N; n++)", "for (int n = 0; n < 1; n++)"),
    ("bwd_bias_drops_last_row", "int or_conv2d_bwd_bias(", "for (int i = 0; i < Ho; i++)", "for (int i = 0; i < Ho - 1; i++)"),
    ("gx_at_ignores_stride", "double or_conv2d_gx_at(", "if (ti < 0 || ti % s) continue;", "if (ti < 0) continue;"),
    ("gw_at_extra_column", "double or_conv2d_gw_at(", "j < j_end && j < Wo", "j <= j_end && j < Wo"),
    ("gb_at_extra_column", "double or_conv2d_gb_at(", "j < j_end && j < Wo", "j <= j_end && j < Wo"),
    ("gb_at_skips_first_column", "double or_conv2d_gb_at(", "for (int j = j_begin;", "for (int j = j_begin + 1;"),
    ("plan_right_halo_short", "static int plan_1d(", "last - e.in_end + 1", "last - e.in_end"),
    ("plan_owned_cols_shifted", "static int plan_1d(", "e.out_begin = r * L / s;", "e.out_begin = r * L / s + (r > 0);"),
    ("halo_drops_first_column", "int or_halo_extend(", "col >= 0 && col < d->W)", "col > 0 && col < d->W)"),
    ("halo_drops_first_row", "int or_halo_extend(", "(row >= 0 && row < d->H", "(row > 0 && row < d->H"),
    ("row_plan_ignores_kernel_height", "int or_shard_plan_h(", "plan_1d(d->H, d->kh,", "plan_1d(d->H, d->kh - 1,"),
    ("sharded_fwd_no_row_crop", "int or_sharded_fwd(", "i + crop_h, t + crop", "i, t + crop"),
    ("sharded_fwd_no_crop", "int or_sharded_fwd(", "+ p) / s;", "+ 0) / s;"),
    ("sharded_bwd_keeps_halo_grads", "int or_sharded_bwd(", "col >= 0 && col < d->W)", "col >= e.in_begin && col < e.in_end)"),
    ("sharded_bwd_keeps_halo_row_grads", "int or_sharded_bwd(", "if (row >= 0 && row < d->H &&", "if (row >= f.in_begin && row < f.in_end &&"),
    ("ln_unbiased_variance", "void or_layernorm_c_fwd(", "var /= C;", "var /= (C - 1);"),
    ("ln_bwd_drops_mean_term", "void or_layernorm_c_bwd(", "gx[o] = rs * (gy[o] * gamma[c] - mg - xh * mgx);", "gx[o] = rs * (gy[o] * gamma[c] - xh * mgx);"),
    ("gelu_missing_sqrt2", "void or_gelu_fwd(", "erf(x[i] / sqrt(2.0))", "erf(x[i])"),
    ("gelu_bwd_drops_density_term", "void or_gelu_bwd(", "(Phi + x[i] * phi)", "(Phi)"),
    ("layerscale_bwd_wrong_gamma_grad", "void or_layerscale_residual_bwd(", "ggamma[c] += branch[o] * gy[o];", "ggamma[c] += gy[o];"),
    ("splitmix_wrong_final_shift", "uint64_t or_splitmix64(", "return z ^ (z >> 31);", "return z ^ (z >> 30);"),
    ("splitmix_counter_off_by_one", "uint64_t or_splitmix64(", "(i + 1) *", "i *"),
    ("drop_path_inverted_keep", "int or_drop_path_mask(", "u >= t ? scale : 0.0f", "u < t ? scale : 0.0f"),
    ("drop_path_unscaled", "int or_drop_path_mask(", "const float scale = 1.0f / (1.0f - p);", "const float scale = 1.0f;"),
    ("drop_path_low_bits", "int or_drop_path_mask(", "offset + (uint64_t)n) >> 40)", "offset + (uint64_t)n) & 0xFFFFFF)"),
    ("droppath_fwd_ignores_mask", "void or_layerscale_droppath_fwd(", "res[o] + mask[n] * gamma[c] * branch[o]", "res[o] + gamma[c] * branch[o]"),
    ("droppath_bwd_gamma_grad_ignores_mask", "void or_layerscale_droppath_bwd(", "ggamma[c] += mask[n] * branch[o] * gy[o];", "ggamma[c] += branch[o] * gy[o];"),
]


def _mutate(src: str, func: str, old: str, new: str) -> str:
    start = src.index(func)
    nxt = src.find("\n}\n", start)
    body = src[start:nxt]
    assert old in body, (func, old)
    return src[:start] + body.replace(old, new, 1) + src[nxt:]


@pytest.mark.parametrize("name,func,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, func, old, new):
    src = open(oracle.SRC).read()
    mutated = _mutate(src, func, old, new)
    assert mutated != src
    cpath = os.path.join(tmp_path, "mutant.c")
    open(cpath, "w").write(mutated)
    lib = oracle.compile_oracle(cpath, os.path.join(tmp_path, "libmutant.so"), openmp=False)
    m = oracle.Oracle(lib)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(m)
        except AssertionError:
            caught.append(pin.__name__)
            break
    assert caught, f"mutant {name} passed every pin"
