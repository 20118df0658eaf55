"""Seeded input generators (no GPU): shapes, normalisation, shards, bf16 rounding."""
import numpy as np
import pytest

import workloads


@pytest.mark.parametrize("name", ["tiny2d", "encoder2d", "decoder2d", "encoder2d_bwd",
                                  "volume3d_bwd"])
def test_shapes_and_weight_normalisation(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w)
    B, Nin, M, D = inp["value"].shape
    assert (B, Nin, M, D) == (w.B, w.Nin, w.M, w.D)
    assert inp["sampling_locations"].shape == (w.B, w.Nq, w.M, w.L, w.P, w.ndim)
    assert inp["sampling_locations"].dtype == np.float32
    a = inp["attention_weights"]
    assert a.shape == (w.B, w.Nq, w.M, w.L, w.P) and a.dtype == np.float32
    assert np.all(a >= 0) and np.all(a <= 1)
    np.testing.assert_allclose(a.reshape(w.B, w.Nq, w.M, -1).sum(-1), 1.0, atol=1e-6)
    ls = inp["level_start_index"]
    sizes = np.prod(inp["spatial_shapes"], axis=1)
    assert ls[0] == 0 and np.all(ls[1:] == np.cumsum(sizes)[:-1]) and sizes.sum() == Nin


def test_named_sizes():
    W = workloads.WORKLOADS
    assert W["encoder2d"].Nin == 19947 and W["encoder2d"].samples == 5_106_432
    assert W["decoder2d"].samples == 307_200
    assert W["volume3d"].Nin == 299_520 and W["volume3d"].samples == 4_194_304
    assert W["tiny2d"].samples == 512


def test_out_of_range_pushes():
    w = workloads.WORKLOADS["encoder2d_bwd"].with_(B=1)
    inp = workloads.make_inputs(w)
    frac = workloads.out_of_range_fraction(w, inp["sampling_locations"])
    assert 0.10 <= frac <= 0.25


def test_bf16_rounding_is_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.0 - 2 ** -8, 3.0e38],
                 dtype=np.float32)
    got = workloads.bf16_bits_to_f32(workloads.f32_to_bf16_bits(x))
    # ties go to the even mantissa
    assert got[1] == 1.0 and got[2] == 1.0 + 4 * 2 ** -8 and got[3] == -2.0
    assert np.isfinite(got[4])


@pytest.mark.parametrize("total,world", [(0, 1), (5, 2), (19947, 8), (7, 7), (3, 4)])
def test_shards_cover_every_unit_once(total, world):
    seen = []
    for r in range(world):
        a, b = workloads.shard_range(total, r, world)
        assert 0 <= a <= b <= total
        seen.extend(range(a, b))
    assert seen == list(range(total))
