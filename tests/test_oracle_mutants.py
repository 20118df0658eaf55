"""Plant plausible mistakes in copies of the oracle; some pin must catch each one.

The mistakes are planted in the oracle's C source on the CPU (a temporary copy), never
in the CUDA path.  A mutant that survives every pin would mean the pins leave that part
of the oracle unchecked.
"""
import os

import pytest

import oracle
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "msda_oracle.c")

# (id, text in the source, replacement, occurrence to change: int index or "all").
# Every mutant keeps its memory accesses inside the arrays it is given.
MUTANTS = [
    ("pixel_offset_sign", "loc[2 * s + 0] * (double)W - 0.5", "loc[2 * s + 0] * (double)W + 0.5", 0),
    ("no_half_pixel_y", "loc[2 * s + 1] * (double)H - 0.5", "loc[2 * s + 1] * (double)H", 0),
    ("swapped_extents_2d", "int64_t H = shapes[2 * l + 0], W = shapes[2 * l + 1];",
     "int64_t W = shapes[2 * l + 0], H = shapes[2 * l + 1];", 0),
    ("corner_weight_flipped", "double wx = dx ? fx : 1.0 - fx;", "double wx = dx ? 1.0 - fx : fx;", 0),
    ("transposed_flattening", "level_start[l] + t[c].h * W + t[c].w",
     "level_start[l] + t[c].w * H + t[c].h", 0),
    ("level_start_dropped", "int64_t row = level_start[l] + t[c].h * W + t[c].w;",
     "int64_t row = t[c].h * W + t[c].w;", 0),
    ("bounds_off_by_one", "t[c].w >= 0 && t[c].w < W);", "t[c].w >= 0 && t[c].w <= W - 2);", 0),
    ("partial_oob_dropped", "if (!(x > -1.0 && x < (double)W", "if (!(x > 0.0 && x < (double)W", 0),
    ("attention_dropped_fwd", "o[d] += a * t[c].wgt * v[d];", "o[d] += t[c].wgt * v[d];", 0),
    ("fy_sign", "double fx = x - x0, fy = y - y0;", "double fx = x - x0, fy = y0 - y;", 0),
    ("head_index_wrong", "const double *v = value + ((b * Nin + row) * M + m) * D;",
     "const double *v = value + ((b * Nin + row) * M + (M - 1 - m)) * D;", 0),
    # backward
    ("grad_loc_wrong_extent", "grad_loc[2 * s + 0] = gx * (double)W;",
     "grad_loc[2 * s + 0] = gx * (double)H;", 0),
    ("grad_loc_sign", "double dwx = dx ? 1.0 : -1.0; /* d wx / d x */",
     "double dwx = dx ? -1.0 : 1.0; /* d wx / d x */", 0),
    ("grad_value_missing_A", "gv[d] += a * t[c].wgt * g[d];", "gv[d] += t[c].wgt * g[d];", 0),
    ("grad_attn_extra_A", "gA += t[c].wgt * gdotv;", "gA += a * t[c].wgt * gdotv;", 0),
    ("grad_y_uses_dwdx", "gy += a * t[c].dwdy * gdotv;", "gy += a * t[c].dwdx * gdotv;", 0),
    # 3D
    ("z_extent_wrong", "double z = loc[3 * s + 2] * (double)Z - 0.5;",
     "double z = loc[3 * s + 2] * (double)H - 0.5;", 0),
    ("transposed_flattening_3d", "(t[c].z * H + t[c].h) * W + t[c].w",
     "(t[c].h * Z + t[c].z) * W + t[c].w", 0),
    ("wz_uses_fy", "double wz = dz ? fz : 1.0 - fz;", "double wz = dz ? fz : 1.0 - fy;", 0),
    ("z_bounds_too_strict", "t[c].inside = (t[c].z >= 0 && t[c].z < Z &&",
     "t[c].inside = (t[c].z >= 0 && t[c].z < Z - 1 &&", 0),
    ("grad_z_wrong_extent", "grad_loc[3 * s + 2] = gz * (double)Z;",
     "grad_loc[3 * s + 2] = gz * (double)W;", 0),
    ("grad_value_3d_missing_A", "gv[d] += a * t[c].wgt * g[d];", "gv[d] += t[c].wgt * g[d];", 1),
]


def _mutate(text, old, new, which):
    n = text.count(old)
    assert n > 0, f"mutation anchor not found: {old!r}"
    if which == "all":
        return text.replace(old, new)
    idx = -1
    for _ in range(which + 1):
        idx = text.index(old, idx + 1)
    return text[:idx] + new + text[idx + len(old):]


@pytest.mark.parametrize("mid,old,new,which", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, mid, old, new, which):
    src = open(SRC).read()
    mutated = _mutate(src, old, new, which)
    assert mutated != src
    csrc = tmp_path / f"mutant_{mid}.c"
    csrc.write_text(mutated)
    lib = oracle.load_library(oracle.compile_source(str(csrc), str(tmp_path / f"{mid}.so")))
    with pytest.raises(AssertionError):
        pins.pin_all(lib, quick=True)


def test_unmutated_oracle_passes_all_pins(tmp_path):
    csrc = tmp_path / "clean.c"
    csrc.write_text(open(SRC).read())
    lib = oracle.load_library(oracle.compile_source(str(csrc), str(tmp_path / "clean.so")))
    pins.pin_all(lib, quick=True)
