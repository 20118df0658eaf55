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
