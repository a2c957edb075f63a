"""Pins of the f64 NeoX RoPE oracle (oracle/rope.py) to the page
"rope_neox_backward.wgsl" (rullama 0.2.0) and to properties of rotations.

* golden cases (tests/golden/rope_neox.json): unit vectors turned by whole
  radians, compared with printed cosines and sines;
* the inverse undoes the forward rotation; rotations at positions p and p'
  compose to the rotation at p + p' (theta is linear in the position);
* the dot product of a rotated query and key depends only on the position
  difference (the point of rotary embeddings);
* every rotated pair keeps its length; dims past 2 * (rope_dims // 2) and
  rope_dims = 0 stay untouched; pos = 0 is the identity;
* a factor table divides the angles: factors 2 at position 2p equal no
  factors at position p;
* each pair (a, b) turns like the complex number a + ib times e^(i theta).
"""
import json
import os

import numpy as np
import pytest

from oracle import rope

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rope_neox.json")


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["what"][:40])
def test_golden(case):
    x = np.array(case["x"], dtype=np.float64).reshape(1, 1, 1, case["head_dim"])
    got = rope.rope_neox(x, case["rope_dims"], case["pos"], case["base"], inverse=case["inverse"])
    np.testing.assert_allclose(got.ravel(), case["expect"], rtol=0, atol=1e-12)


@pytest.mark.parametrize("rope_dims", [2, 8, 62, 64])
def test_inverse_undoes_forward(rope_dims):
    x = rand((2, 3, 17, 64), 1)
    y = rope.rope_neox(x, rope_dims, 5, 10000.0)
    back = rope.rope_neox(y, rope_dims, 5, 10000.0, inverse=True)
    np.testing.assert_allclose(back, x, rtol=0, atol=1e-12)


def test_rotations_compose_additively_in_position():
    x = rand((1, 2, 1, 16), 2)
    twice = rope.rope_neox(rope.rope_neox(x, 16, 7, 500.0), 16, 11, 500.0)
    once = rope.rope_neox(x, 16, 18, 500.0)
    np.testing.assert_allclose(twice, once, rtol=0, atol=1e-11)


def test_dot_product_depends_only_on_the_position_difference():
    q = rand((1, 1, 1, 32), 3)
    k = rand((1, 1, 1, 32), 4)
    ref = None
    for shift in (0, 1, 13, 250):
        qr = rope.rope_neox(q, 32, 40 + shift, 10000.0)
        kr = rope.rope_neox(k, 32, 33 + shift, 10000.0)
        dot = float((qr * kr).sum())
        ref = dot if ref is None else ref
        assert abs(dot - ref) < 1e-11
    # and it does depend on the difference
    qr = rope.rope_neox(q, 32, 41, 10000.0)
    kr = rope.rope_neox(k, 32, 33, 10000.0)
    assert abs(float((qr * kr).sum()) - ref) > 1e-3


def test_pairs_keep_their_length_and_the_rest_is_untouched():
    x = rand((2, 2, 9, 20), 5)
    for rope_dims in (0, 1, 7, 12, 20):
        y = rope.rope_neox(x, rope_dims, 3, 777.0)
        half = rope_dims // 2
        np.testing.assert_array_equal(y[..., 2 * half:], x[..., 2 * half:])
        for i in range(half):
            np.testing.assert_allclose(np.hypot(y[..., i], y[..., i + half]),
                                       np.hypot(x[..., i], x[..., i + half]), rtol=1e-13)


def test_position_zero_is_the_identity():
    x = rand((1, 2, 1, 8), 6)
    np.testing.assert_array_equal(rope.rope_neox(x, 8, 0, 10000.0), x)


def test_patch_n_sits_at_position_pos0_plus_n():
    x = rand((1, 2, 5, 8), 7)
    y = rope.rope_neox(x, 8, 10, 10000.0)
    for n in range(5):
        one = rope.rope_neox(x[:, :, n:n + 1, :], 8, 10 + n, 10000.0)
        np.testing.assert_array_equal(y[:, :, n:n + 1, :], one)


def test_factors_divide_the_angles():
    x = rand((1, 1, 3, 12), 8)
    with_f = rope.rope_neox(x, 12, 2 * 9, 10000.0, factors=np.full(6, 2.0))
    without = rope.rope_neox(x, 12, 9, 10000.0)
    # positions 18, 19, 20 with factor 2 = positions 9, 9.5, 10 without: only patch 0 matches
    np.testing.assert_allclose(with_f[:, :, 0], without[:, :, 0], rtol=0, atol=1e-12)


def test_pairs_turn_like_complex_multiplication():
    x = rand((1, 1, 4, 10), 9)
    theta = rope.angles(4, 10, 3, 250.0)
    z = (x[..., :5] + 1j * x[..., 5:10]) * np.exp(1j * theta)[None, None]
    y = rope.rope_neox(x, 10, 3, 250.0)
    np.testing.assert_allclose(y[..., :5], z.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(y[..., 5:10], z.imag, rtol=0, atol=1e-12)


def test_frequency_schedule_of_the_page():
    # theta_i = pos * base^(-2i / rope_dims): for rope_dims 8 and base 10^4 the
    # pairs have frequencies 1, 10^-1, 10^-2, 10^-3
    theta = rope.angles(1, 8, 3, 10000.0)
    np.testing.assert_allclose(theta[0], [3.0, 0.3, 0.03, 0.003], rtol=1e-13)
