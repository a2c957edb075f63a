"""Pins for the f64 oracle, checked against things other than itself.

Each pin is chosen so that a plausible slip in the oracle fails at least one:

* closed forms (tests/golden/closed_form.json): a stray 1/sqrt(head_dim), a
  swapped q/k/v operand, a wrong head or batch stride, a missing max
  subtraction (overflow at scores near 1000), a wrong normaliser;
* invariants of softmax(q k^T) v: one patch gives v; identical keys give the
  mean of v; permuting (key, value) rows together changes nothing; a dominant
  score selects its value row; a shared key offset changes nothing; rows are
  convex combinations of value rows; the map is linear in v; each output row
  depends only on its own query row;
* a library routine: scipy.special.softmax followed by a numpy product;
* brute force on tiny inputs at 60 significant digits (mpmath), without the
  max subtraction.

The quantity pinned is what the WGSL shader vision_attention_flash_sub_hpd_f16
(rullama 0.1.0) writes: out = o / l of its online softmax over all keys.
"""
import json
import math
import os

import numpy as np
import pytest

from vattn_inputs import WORKLOADS, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form.json")


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _eval_expected(tree):
    env = {name: getattr(math, name) for name in dir(math) if not name.startswith("_")}
    if isinstance(tree, list):
        return [_eval_expected(t) for t in tree]
    return float(eval(tree, {"__builtins__": {}}, env))  # noqa: S307 (fixture text)


def _load_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _load_cases(), ids=lambda c: c["name"])
def test_closed_forms(oracle_mod, case):
    q, k, v = _f32(case["q"]), _f32(case["k"]), _f32(case["v"])
    assert list(q.shape) == case["shape"]
    expected = np.asarray(_eval_expected(case["expected"]), dtype=np.float64)
    out = oracle_mod.forward(q, k, v, threads=2)
    assert out.shape == expected.shape
    np.testing.assert_allclose(out, expected, rtol=0, atol=case["atol"])


def _rand(shape, seed, scale=1.0):
    q, k, v = make_inputs(*shape, seed=seed)
    return q * np.float32(scale), k, v


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_single_patch_gives_v(oracle_mod, seed):
    q, k, v = _rand((2, 3, 1, 17), seed, scale=40.0)
    out = oracle_mod.forward(q, k, v)
    np.testing.assert_array_equal(out, v.astype(np.float64))


@pytest.mark.parametrize("seed", [4, 5])
def test_identical_keys_give_mean_of_v(oracle_mod, seed):
    q, k, v = _rand((1, 2, 37, 8), seed, scale=3.0)
    k[:] = k[:, :, :1, :]  # every key row equal to row 0 of its head
    out = oracle_mod.forward(q, k, v)
    mean = v.astype(np.float64).mean(axis=2, keepdims=True)
    np.testing.assert_allclose(out, np.broadcast_to(mean, out.shape), rtol=0, atol=1e-13)


@pytest.mark.parametrize("seed", [6, 7])
def test_joint_key_value_permutation_is_invisible(oracle_mod, seed):
    q, k, v = _rand((2, 2, 50, 12), seed, scale=2.0)
    perm = np.random.Generator(np.random.PCG64(seed)).permutation(50)
    out = oracle_mod.forward(q, k, v)
    out_p = oracle_mod.forward(q, _f32(k[:, :, perm]), _f32(v[:, :, perm]))
    np.testing.assert_allclose(out_p, out, rtol=0, atol=1e-13)


def test_permuting_values_alone_is_visible(oracle_mod):
    # guards the previous test: it must not pass because v is ignored
    q, k, v = _rand((1, 1, 20, 4), 8, scale=4.0)
    perm = np.roll(np.arange(20), 1)
    out = oracle_mod.forward(q, k, v)
    out_p = oracle_mod.forward(q, k, _f32(v[:, :, perm]))
    assert np.abs(out_p - out).max() > 1e-2


def test_dominant_score_selects_its_value_row(oracle_mod):
    # keys are the unit vectors e_j (in a shuffled order); query i is 60 along
    # its target key's direction plus noise in [-1, 1], so its target score
    # beats every other score by at least 58 - 2 = 56 > 40
    N = D = 24
    rng = np.random.Generator(np.random.PCG64(9))
    order = rng.permutation(N)
    k = np.zeros((1, 1, N, D))
    k[0, 0, np.arange(N), order] = 1.0
    targets = rng.integers(0, N, size=N)
    q = rng.uniform(-1.0, 1.0, size=(1, 1, N, D))
    q[0, 0, np.arange(N), order[targets]] += 60.0
    v = rng.standard_normal((1, 1, N, D))
    q, k, v = _f32(q), _f32(k), _f32(v)
    out = oracle_mod.forward(q, k, v)[0, 0]
    for i in range(N):
        s = q[0, 0, i, order].astype(np.float64)  # score of key j is q[i, order[j]]
        j = targets[i]
        gap = s[j] - np.max(np.delete(s, j))
        assert gap >= 40.0
        bound = (N - 1) * math.exp(-gap) * 2 * np.abs(v).max()
        np.testing.assert_allclose(out[i], v[0, 0, j].astype(np.float64), rtol=0,
                                   atol=max(bound, 1e-15))


def test_shared_key_offset_changes_nothing(oracle_mod):
    q, k, v = _rand((1, 3, 40, 16), 10)
    c = np.random.Generator(np.random.PCG64(11)).standard_normal((1, 3, 1, 16)) * 2
    k2 = _f32(k + c)
    # adding c to every key adds q_i . c to every score of row i, which the
    # softmax removes; what remains is the f32 rounding of k + c
    out = oracle_mod.forward(q, k, v)
    out2 = oracle_mod.forward(q, k2, v)
    np.testing.assert_allclose(out2, out, rtol=0, atol=2e-5)


def test_zero_query_gives_mean(oracle_mod):
    _, k, v = _rand((2, 2, 33, 5), 12)
    q = np.zeros_like(k)
    out = oracle_mod.forward(q, k, v)
    mean = v.astype(np.float64).mean(axis=2, keepdims=True)
    np.testing.assert_allclose(out, np.broadcast_to(mean, out.shape), rtol=0, atol=1e-14)


def test_constant_values_give_constant(oracle_mod):
    q, k, _ = _rand((1, 2, 70, 9), 13, scale=5.0)
    v = np.full_like(q, 1.0)
    out = oracle_mod.forward(q, k, v)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-14)


def test_convex_combination_bounds(oracle_mod):
    q, k, v = _rand((2, 2, 45, 7), 14, scale=3.0)
    out = oracle_mod.forward(q, k, v)
    lo = v.min(axis=2, keepdims=True).astype(np.float64) - 1e-12
    hi = v.max(axis=2, keepdims=True).astype(np.float64) + 1e-12
    assert np.all(out >= lo) and np.all(out <= hi)


def test_linear_in_values(oracle_mod):
    q, k, v1 = _rand((1, 2, 30, 6), 15, scale=2.0)
    v2 = make_inputs(1, 2, 30, 6, seed=16)[2]
    a, b = 0.75, -2.5  # exact in f32 together with the sums below
    out1 = oracle_mod.forward(q, k, v1)
    out2 = oracle_mod.forward(q, k, v2)
    v3 = _f32(a * v1.astype(np.float64) + b * v2.astype(np.float64))
    out3 = oracle_mod.forward(q, k, v3)
    ref = a * out1 + b * out2
    # v3 is rounded to f32: allow that rounding (<= 2^-24 relative per entry)
    np.testing.assert_allclose(out3, ref, rtol=0, atol=1e-6)


def test_rows_depend_only_on_their_query(oracle_mod):
    q, k, v = _rand((1, 1, 25, 8), 17)
    out = oracle_mod.forward(q, k, v)
    q2 = q.copy()
    q2[0, 0, 3] += 1.0
    out2 = oracle_mod.forward(q2, k, v)
    changed = np.abs(out2 - out).max(axis=-1)[0, 0]
    assert changed[3] > 1e-3
    assert np.all(np.delete(changed, 3) == 0.0)


@pytest.mark.parametrize("shape", [(1, 1, 5, 3), (2, 3, 17, 8), (1, 2, 129, 72)])
def test_matches_scipy_softmax(oracle_mod, shape):
    from scipy.special import softmax
    q, k, v = _rand(shape, 18, scale=2.0)
    s = q.astype(np.float64) @ np.swapaxes(k.astype(np.float64), -1, -2)
    ref = softmax(s, axis=-1) @ v.astype(np.float64)
    out = oracle_mod.forward(q, k, v)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape,scale", [((1, 1, 3, 2), 1.0), ((1, 2, 4, 3), 6.0),
                                         ((2, 1, 5, 4), 20.0)])
def test_brute_force_high_precision(oracle_mod, shape, scale):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60
    q, k, v = _rand(shape, 19, scale=scale)
    out = oracle_mod.forward(q, k, v)
    B, H, N, D = shape
    for b in range(B):
        for h in range(H):
            for i in range(N):
                w = [mpmath.exp(mpmath.fsum(mpmath.mpf(float(q[b, h, i, d])) *
                                            mpmath.mpf(float(k[b, h, j, d]))
                                            for d in range(D)))
                     for j in range(N)]
                tot = mpmath.fsum(w)
                for d in range(D):
                    ref = mpmath.fsum(w[j] * mpmath.mpf(float(v[b, h, j, d]))
                                      for j in range(N)) / tot
                    assert abs(out[b, h, i, d] - float(ref)) <= 1e-13


def test_rows_entry_matches_full(oracle_mod):
    q, k, v = _rand((2, 3, 41, 10), 20)
    full = oracle_mod.forward(q, k, v).reshape(-1, 10)
    idx = np.array([0, 5, 40, 41, 100, 245, 2 * 3 * 41 - 1])
    np.testing.assert_array_equal(oracle_mod.rows(q, k, v, idx), full[idx])


def test_thread_count_does_not_change_results(oracle_mod):
    q, k, v = _rand((1, 2, 64, 32), 21)
    a = oracle_mod.forward(q, k, v, threads=1)
    b = oracle_mod.forward(q, k, v, threads=7)
    np.testing.assert_array_equal(a, b)


def test_empty_problems_are_no_ops(oracle_mod):
    for shape in [(0, 2, 4, 8), (1, 0, 4, 8), (1, 2, 0, 8)]:
        z = np.zeros(shape, dtype=np.float32)
        assert oracle_mod.forward(z, z, z).shape == shape


def test_workload_generator_recipe():
    # determinism, dtype, scaling and the shared per-head offset
    w = WORKLOADS[5]
    q, k, v = make_inputs(2, 3, 500, 64, seed=w.seed, peaked=True)
    q2, _, _ = make_inputs(2, 3, 500, 64, seed=w.seed, peaked=True)
    np.testing.assert_array_equal(q, q2)
    assert q.dtype == k.dtype == v.dtype == np.float32
    assert abs(q.std() * 8.0 - 1.0) < 0.02  # q scaled by 1/sqrt(64)
    assert abs(v.std() - 1.0) < 0.02
    # same offset for both batch entries of a head, different across heads
    km = k.astype(np.float64).mean(axis=2)
    assert np.abs(km[0] - km[1]).max() < 0.25
    assert np.abs(km[0, 0] - km[0, 1]).max() > 0.5
    off_var = km.var()
    assert 1.2 < off_var < 3.0  # variance-2 offsets (std sqrt 2)
    assert {i: WORKLOADS[i].shape for i in WORKLOADS} == {
        1: (1, 2, 64, 32), 2: (1, 16, 256, 64), 3: (4, 16, 1024, 64),
        4: (1, 16, 4100, 72), 5: (8, 16, 2304, 64)}
