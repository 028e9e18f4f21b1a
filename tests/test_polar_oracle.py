"""Pins of the polar-angle quantizer oracle (oracle/polar_oracle.py) to
facts that do not come from the oracle itself: the norm that the tree keeps
exactly, vectors built on the grid that must come back unchanged, the
nearest grid point at d = 2 by brute force, a unit vector whose angles are
all zero, and the packed layout's round trip."""
import math

import numpy as np
import pytest

from oracle import polar_oracle as P


@pytest.mark.parametrize("d", [2, 4, 32, 64, 128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_decoded_norm_is_the_stored_radius(d, bits):
    """cos^2 + sin^2 = 1 at every node: the decoded vector's norm equals the
    stored fp16 radius whatever the angles."""
    x = np.random.default_rng(d * 10 + bits).standard_normal((64, d))
    idx, r16 = P.polar_encode(x, bits)
    y = P.polar_decode(idx, r16, bits)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), r16.astype(np.float64), rtol=1e-12, atol=0)
    # and the radius is the vector's norm, rounded to fp16
    assert np.array_equal(r16, np.linalg.norm(x, axis=1).astype(np.float16))


@pytest.mark.parametrize("d", [4, 16, 128])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_vectors_on_the_grid_come_back(d, bits):
    """A vector built from grid angles (levels above the first take grid
    points in [0, pi/2], as radii are non-negative) and an fp16 radius is
    encoded to exactly those indices and decoded to itself."""
    rng = np.random.default_rng(7 * d + bits)
    steps = (1 << bits) - 1
    grid = np.array([k / steps * 2 * math.pi - math.pi for k in range(steps + 1)])
    low = [k for k in range(steps + 1) if 0.0 <= grid[k] <= math.pi / 2]
    N = 32
    idx = np.zeros((N, d - 1), dtype=np.int64)
    idx[:, :d // 2] = rng.integers(0, steps + 1, size=(N, d // 2))
    idx[:, d // 2:] = rng.choice(low, size=(N, d - 1 - d // 2))
    r16 = rng.uniform(0.5, 4.0, size=N).astype(np.float16)
    x = P.polar_decode(idx, r16, bits)
    idx2, r2 = P.polar_encode(x, bits)
    assert np.array_equal(idx2, idx)
    assert np.array_equal(r2, r16)
    np.testing.assert_allclose(P.polar_decode(idx2, r2, bits), x, rtol=0, atol=1e-12)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_two_values_take_the_nearest_grid_angle(bits):
    """At d = 2 the index is the grid point nearest atan2(x1, x0), found by
    brute force over the 2^b points (the page's round on [-pi, pi])."""
    x = np.random.default_rng(bits).standard_normal((2000, 2))
    idx, _ = P.polar_encode(x, bits)
    theta = np.arctan2(x[:, 1], x[:, 0])
    steps = (1 << bits) - 1
    grid = np.array([k / steps * 2 * math.pi - math.pi for k in range(steps + 1)])
    near = np.argmin(np.abs(theta[:, None] - grid[None, :]), axis=1)
    assert np.array_equal(idx[:, 0], near)


@pytest.mark.parametrize("bits,want", [(1, 0), (2, 2), (3, 4), (4, 8)])
def test_first_unit_vector(bits, want):
    """e_0: every pair is (r, 0), every angle 0, so every index rounds
    (2^b - 1)/2 half to even; the radius is 1."""
    d = 64
    x = np.zeros((1, d))
    x[0, 0] = 1.0
    idx, r16 = P.polar_encode(x, bits)
    assert np.all(idx == want) and r16[0] == 1.0
    th = want / ((1 << bits) - 1) * 2 * math.pi - math.pi
    y = P.polar_decode(idx, r16, bits)
    # the first coordinate is the product of the cosines down the left edge
    assert abs(y[0, 0] - math.cos(th) ** 6) < 1e-12


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_packed_indices_round_trip(bits):
    d = 128
    idx = np.random.default_rng(bits + 40).integers(0, 1 << bits, size=(16, d - 1))
    packed = P.pack_polar(idx, bits)
    assert packed.shape == (16, d * bits // 8)
    assert np.array_equal(P.unpack_polar(packed, bits, d), idx)


def test_error_falls_with_bits():
    u = np.random.default_rng(3).standard_normal((500, 128))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    mse = []
    for bits in (1, 2, 3, 4):
        idx, r16 = P.polar_encode(u, bits)
        mse.append(np.mean(np.sum((P.polar_decode(idx, r16, bits) - u) ** 2, axis=1)))
    assert all(a > b for a, b in zip(mse, mse[1:])), mse
