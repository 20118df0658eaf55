"""The CPU oracle against its pins (no GPU).  See ``oracle_pins.py`` for what each pins."""
import numpy as np
import pytest

import oracle_pins as pins


def test_golden_bilinear_worked_example(oracle_mod):
    pins.pin_golden_2d()


def test_golden_trilinear_cube_corners(oracle_mod):
    pins.pin_golden_3d()


@pytest.mark.parametrize("nd", [2, 3])
def test_dense_tent_kernel_brute_force(oracle_mod, nd):
    pins.pin_dense(nd)


def test_dense_brute_force_on_tiny_workload(oracle_mod):
    pins.pin_dense_tiny_workload()


@pytest.mark.parametrize("nd", [2, 3])
def test_constant_map_returns_constant(oracle_mod, nd):
    pins.pin_constant_map(nd)


def test_exact_gather_at_pixel_centres(oracle_mod):
    pins.pin_exact_gather()


@pytest.mark.parametrize("nd", [2, 3])
def test_linearity_and_level_isolation(oracle_mod, nd):
    pins.pin_linearity_and_levels(nd)


def test_single_slice_3d_equals_2d(oracle_mod):
    pins.pin_3d_single_slice_is_2d()


@pytest.mark.parametrize("nd", [2, 3])
def test_non_finite_locations_contribute_nothing(oracle_mod, nd):
    pins.pin_nonfinite_locations(nd)


@pytest.mark.parametrize("nd", [2, 3])
def test_backward_matches_finite_differences(oracle_mod, nd):
    pins.pin_backward_finite_differences(nd)


@pytest.mark.parametrize("nd", [2, 3])
def test_backward_adjoint_identities(oracle_mod, nd):
    pins.pin_adjoint_identities(nd)


@pytest.mark.parametrize("nd", [2, 3])
def test_zero_padding_gradients(oracle_mod, nd):
    pins.pin_zero_padding_gradients(nd)


def test_backward_finite_differences_on_encoder_query_slice(oracle_mod):
    """One query of the encoder-shaped backward workload (all heads, levels, points)."""
    import workloads
    w = workloads.WORKLOADS["encoder2d_bwd"]
    inp = workloads.make_inputs(w)
    q = 777
    case = dict(value=inp["value"][:1].astype(np.float64),
                spatial_shapes=inp["spatial_shapes"],
                level_start_index=inp["level_start_index"],
                sampling_locations=inp["sampling_locations"][:1, q:q + 1].astype(np.float64),
                attention_weights=inp["attention_weights"][:1, q:q + 1].astype(np.float64),
                grad_out=inp["grad_out"][:1, q:q + 1].astype(np.float64))
    pins.pin_backward_finite_differences(2, case=case)


def test_adjoint_identities_at_encoder_size(oracle_mod):
    import workloads
    w = workloads.WORKLOADS["encoder2d_bwd"]
    inp = workloads.make_inputs(w)
    case = {k: inp[k] for k in ("value", "spatial_shapes", "level_start_index",
                                "sampling_locations", "attention_weights", "grad_out")}
    pins.pin_adjoint_identities(2, case=case)


# ---------------------------------------------------------------- probability-aware pruning

def test_pruned_oracle_reduces_to_the_plain_core_and_to_zero(oracle_mod):
    import workloads
    for nd, shapes in ((2, [(9, 11), (4, 6)]), (3, [(4, 5, 6), (2, 2, 3)])):
        inp = workloads.random_problem(nd, shapes, B=2, Nq=30, M=2, D=8, P=4, seed=41,
                                       backward=False)
        args = (nd, inp["value"], inp["spatial_shapes"], inp["level_start_index"],
                inp["sampling_locations"], inp["attention_weights"])
        plain = oracle_mod.forward(*args)
        assert np.array_equal(oracle_mod.forward_pruned(*args, 0.0), plain)
        big = float(np.abs(inp["attention_weights"]).max()) * 2
        assert np.all(oracle_mod.forward_pruned(*args, big) == 0.0)
        assert np.all(oracle_mod.pruning_bound(*args, 0.0) == 0.0)


def test_pruning_error_stays_within_its_bound_and_the_bound_is_tight(oracle_mod):
    import workloads
    inp = workloads.random_problem(2, [(9, 11), (4, 6)], B=2, Nq=50, M=3, D=8, P=4, seed=42,
                                   backward=False)
    args = (2, inp["value"], inp["spatial_shapes"], inp["level_start_index"],
            inp["sampling_locations"], inp["attention_weights"])
    plain = oracle_mod.forward(*args)
    for tau in (0.02, 0.05, 0.1):
        err = np.abs(oracle_mod.forward_pruned(*args, tau) - plain)
        bound = oracle_mod.pruning_bound(*args, tau)
        assert np.all(err <= bound + 1e-12)
        assert bound.max() > 0
    # tight case: the only dropped sample sits exactly on pixel (3, 3) (corner weights
    # 1, 0, 0, 0) and that pixel holds the largest value of its cell, so the error equals
    # the bound
    H = W = 8
    value = np.abs(np.random.default_rng(43).standard_normal((1, H * W, 1, 4))) + 0.5
    value[0, 3 * W + 3] += 10.0
    loc = np.full((1, 1, 1, 1, 2, 2), (3 + 0.5) / 8)
    attn = np.array([0.01, 0.99]).reshape(1, 1, 1, 1, 2)
    a2 = (2, value, np.array([[H, W]]), np.array([0]), loc, attn)
    err = np.abs(oracle_mod.forward_pruned(*a2, 0.05) - oracle_mod.forward(*a2))
    assert np.allclose(err, oracle_mod.pruning_bound(*a2, 0.05), rtol=0, atol=1e-15)


# ---------------------------------------------------------------- fused prologue

def test_fused_oracle_softmax_and_locations_on_hand_worked_cases(oracle_mod):
    H, W = 6, 8                                   # not square: a swapped extent shows
    value = np.random.default_rng(50).standard_normal((1, H * W, 1, 4))
    sh, ls = np.array([[H, W]]), np.array([0])
    # reference at the centre of pixel (x=2, y=5); integer pixel offsets (+1, 0) and
    # (-2, -1) land exactly on pixels (3, 5) and (0, 4): exact gathers of those rows
    ref = np.array([(2 + 0.5) / W, (5 + 0.5) / H]).reshape(1, 1, 1, 2)
    off = np.array([[1.0, 0.0], [-2.0, -1.0]]).reshape(1, 1, 1, 1, 2, 2)
    # logits 0 and ln 3: softmax weights 1/4 and 3/4
    logits = np.array([0.0, np.log(3.0)]).reshape(1, 1, 1, 1, 2)
    out = oracle_mod.forward_fused(2, value, sh, ls, ref, off, logits)
    want = 0.25 * value[0, 5 * W + 3, 0] + 0.75 * value[0, 4 * W + 0, 0]
    assert np.allclose(out.reshape(-1), want, rtol=0, atol=1e-6)
    assert np.allclose(oracle_mod.softmax_weights(logits).reshape(-1), [0.25, 0.75],
                       rtol=0, atol=1e-15)
    # two levels with one point each: the softmax runs across levels (weights 1/4, 3/4),
    # and each level's offset is in that level's pixels (level 1 is 3 x 4: pixel (1, 2))
    sh2 = np.array([[H, W], [3, 4]])
    ls2 = np.array([0, H * W])
    v2 = np.random.default_rng(51).standard_normal((1, H * W + 12, 1, 4))
    ref2 = np.array([[(2 + 0.5) / W, (5 + 0.5) / H], [(0 + 0.5) / 4, (1 + 0.5) / 3]])
    off2 = np.array([[0.0, 0.0], [1.0, 1.0]]).reshape(1, 1, 1, 2, 1, 2)
    out2 = oracle_mod.forward_fused(2, v2, sh2, ls2, ref2.reshape(1, 1, 2, 2), off2,
                                    logits.reshape(1, 1, 1, 2, 1))
    want2 = 0.25 * v2[0, 5 * W + 2, 0] + 0.75 * v2[0, H * W + 2 * 4 + 1, 0]
    assert np.allclose(out2.reshape(-1), want2, rtol=0, atol=1e-6)


def test_fused_oracle_invariants(oracle_mod):
    import workloads
    w = workloads.WORKLOADS["decoder2d"].with_(B=1, Nq=20)
    f = workloads.make_fused_inputs(w)
    args = (2, f["value"], f["spatial_shapes"], f["level_start_index"], f["reference_points"],
            f["sampling_offsets"])
    base = oracle_mod.forward_fused(*args, f["attention_logits"])
    # softmax is invariant to a shift of the logits
    shifted = oracle_mod.forward_fused(*args, f["attention_logits"].astype(np.float64) + 7.0)
    assert np.allclose(shifted, base, rtol=1e-9, atol=1e-12)
    # equal logits give uniform weights: a constant value map returns the constant when
    # every sample lands inside its level (zero offsets at pixel-centre references)
    const = np.full_like(f["value"], 2.5)
    inside = (2, const, f["spatial_shapes"], f["level_start_index"],
              np.full_like(f["reference_points"], 0.5), np.zeros_like(f["sampling_offsets"]))
    out = oracle_mod.forward_fused(*inside, np.zeros_like(f["attention_logits"]))
    assert np.allclose(out, 2.5, rtol=0, atol=1e-12)
    # the weights of every (query, head) sum to one
    a = oracle_mod.softmax_weights(f["attention_logits"])
    assert np.allclose(a.reshape(a.shape[:3] + (-1,)).sum(-1), 1.0, atol=1e-12)


def _fused_case(nd, seed):
    rng = np.random.default_rng(seed)
    shapes = np.array([(5, 7), (3, 4)] if nd == 2 else [(3, 4, 5), (2, 3, 3)], dtype=np.int64)
    L = len(shapes)
    B, Nq, M, P, D = 2, 3, 2, 3, 3
    Nin = int(np.prod(shapes, axis=1).sum())
    starts = np.concatenate([[0], np.cumsum(np.prod(shapes, axis=1))[:-1]])
    return dict(value=rng.standard_normal((B, Nin, M, D)), spatial_shapes=shapes,
                level_start_index=starts,
                reference_points=rng.uniform(0.2, 0.8, (B, Nq, L, nd)).astype(np.float32),
                sampling_offsets=(rng.standard_normal((B, Nq, M, L, P, nd)) * 1.5).astype(
                    np.float32),
                attention_logits=rng.standard_normal((B, Nq, M, L, P)).astype(np.float32),
                grad_out=rng.standard_normal((B, Nq, M * D)), rng=rng)


@pytest.mark.parametrize("nd", [2, 3])
def test_fused_backward_matches_finite_differences_of_the_fused_forward(oracle_mod, nd):
    """The fused prologue's gradients against central differences of forward_fused: in the
    logits (double softmax, small step), in the pixel offsets and in the reference points
    (fp32 locations, a 0.02-pixel step kept inside every sample's cell: the interpolation
    is quadratic along a line there, so the central difference is exact up to rounding),
    and the value adjoint."""
    c = _fused_case(nd, 70 + nd)
    rng = c.pop("rng")
    g = c["grad_out"]
    base = (nd, c["value"], c["spatial_shapes"], c["level_start_index"])
    gv, g_off, g_logit, g_ref = oracle_mod.backward_fused(
        *base, c["reference_points"], c["sampling_offsets"], c["attention_logits"], g)

    def f(ref=None, off=None, z=None):
        out = oracle_mod.forward_fused(
            *base, c["reference_points"] if ref is None else ref,
            c["sampling_offsets"] if off is None else off,
            c["attention_logits"] if z is None else z)
        return float(np.sum(g * out))

    # logits
    dz = rng.standard_normal(c["attention_logits"].shape)
    z0 = c["attention_logits"].astype(np.float64)
    h = 1e-5
    fd = (f(z=z0 + h * dz) - f(z=z0 - h * dz)) / (2 * h)
    an = float(np.sum(g_logit * dz))
    assert abs(fd - an) <= 1e-7 * (1 + abs(an)), (fd, an)
    # offsets and reference points: only coordinates at least 0.1 px from a kink move
    ext = c["spatial_shapes"][:, ::-1].astype(np.float64)[None, None, None, :, None, :]
    loc = oracle_mod.fused_locations(c["spatial_shapes"], c["reference_points"],
                                     c["sampling_offsets"]).astype(np.float64)
    pix = loc * ext - 0.5
    smooth = np.abs(pix - np.round(pix)) > 0.1
    step = 0.02                                                      # pixels
    d_off = np.where(smooth, rng.standard_normal(pix.shape), 0.0)
    o0 = c["sampling_offsets"].astype(np.float64)
    fd = (f(off=(o0 + step * d_off).astype(np.float32)) -
          f(off=(o0 - step * d_off).astype(np.float32))) / (2 * step)
    an = float(np.sum(g_off * d_off))
    mag = float(np.sum(np.abs(g_off * d_off)))
    assert abs(fd - an) <= 2e-3 * (1e-3 + mag), (fd, an)
    # a reference coordinate moves every sample of its (b, q, l) along that axis
    ref_smooth = smooth.all(axis=(2, 4))                             # [B, Nq, L, nd]
    d_ref = np.where(ref_smooth, rng.standard_normal(ref_smooth.shape), 0.0)
    assert d_ref.any()
    hr = step / ext[0, 0, 0, :, 0, :][None, None]                    # 0.02 px in each axis
    r0 = c["reference_points"].astype(np.float64)
    fd = (f(ref=(r0 + hr * d_ref).astype(np.float32)) -
          f(ref=(r0 - hr * d_ref).astype(np.float32))) / (2 * step)
    an = float(np.sum(g_ref * d_ref * hr / step))
    mag = float(np.sum(np.abs(g_ref * d_ref * hr / step)))
    assert abs(fd - an) <= 2e-3 * (1e-3 + mag), (fd, an)
    # value: linear, so the adjoint identity holds exactly up to rounding
    out = oracle_mod.forward_fused(*base, c["reference_points"], c["sampling_offsets"],
                                   c["attention_logits"])
    assert abs(float(np.sum(c["value"] * gv)) - float(np.sum(g * out))) <= 1e-10 * (
        1 + float(np.sum(np.abs(g * out))))


def test_fused_backward_logit_gradients_sum_to_zero(oracle_mod):
    """The softmax is unchanged by adding a constant to an item's logits, so the logit
    gradients of every (query, head) sum to zero."""
    c = _fused_case(2, 80)
    c.pop("rng")
    _, _, g_logit, _ = oracle_mod.backward_fused(
        2, c["value"], c["spatial_shapes"], c["level_start_index"], c["reference_points"],
        c["sampling_offsets"], c["attention_logits"], c["grad_out"])
    s = g_logit.reshape(g_logit.shape[:3] + (-1,)).sum(-1)
    assert np.allclose(s, 0.0, atol=1e-12)


@pytest.mark.parametrize("nd", [2, 3])
def test_multicore_forward_equals_the_serial_forward(oracle_mod, nd):
    """The oracle's all-core forward (used to time it on every host core) cuts the queries
    into blocks and runs the serial forward on each: every output must be bit-identical to
    the serial call, with batch > 1 and a query count that leaves a ragged last block."""
    import workloads
    shapes = [(9, 11), (5, 6)] if nd == 2 else [(4, 5, 6), (2, 3, 3)]
    inp = workloads.random_problem(nd, shapes, B=3, Nq=150, M=3, D=8, P=3, seed=71,
                                   backward=False)
    args = (nd, inp["value"], inp["spatial_shapes"], inp["level_start_index"],
            inp["sampling_locations"], inp["attention_weights"])
    serial = oracle_mod.forward(*args)
    for t in (2, 5, 0):
        assert np.array_equal(oracle_mod.forward(*args, threads=t), serial), t
