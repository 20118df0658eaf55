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
