"""Pins of the f64 conv1d rolling-buffer oracle (oracle/conv1d.py) to the page
"conv1d.wgsl" (cera 0.2.0) and to what a causal depthwise convolution is.

* golden cases (tests/golden/conv1d_step.json): small integers worked by hand
  from the page's formula and buffer layout;
* T steps from an empty (zero) buffer give the causal convolution of each
  channel's input sequence with its taps, computed by numpy.convolve (a
  library routine, a different formulation: the taps of tap index j weigh
  the input j - d_conv steps back);
* after T >= d_conv steps the buffer holds the last d_conv inputs, oldest
  first; a non-zero buffer acts as the d_conv inputs before the first step;
* the step is linear in (input, buffer) and in the weights; taps past d_conv
  are never read; a batch of sequences is the same as one call per sequence;
* kernel_size < d_conv + 1 is refused.
"""
import json
import os

import numpy as np
import pytest

from oracle import conv1d

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "conv1d_step.json")


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["what"][:40])
def test_golden(case):
    h, dc, ks = case["hidden"], case["d_conv"], case["kernel_size"]
    x = np.array(case["input"], np.float64)
    buf = np.array(case["buffer"], np.float64).reshape(dc, h)
    w = np.array(case["weight"], np.float64).reshape(h, ks)
    out, nb = conv1d.conv1d_step(x, buf, w)
    np.testing.assert_array_equal(out, case["out"])
    np.testing.assert_array_equal(nb.ravel(), case["buffer_after"])


def run_steps(xs, buf, w):
    outs = []
    for x in xs:
        o, buf = conv1d.conv1d_step(x, buf, w)
        outs.append(o)
    return np.array(outs), buf


@pytest.mark.parametrize("d_conv,kernel_size", [(0, 1), (1, 2), (2, 3), (3, 4), (3, 6), (7, 8)])
def test_steps_from_zero_equal_causal_convolution(d_conv, kernel_size):
    rng = np.random.default_rng(10 + d_conv)
    T, hidden = 12, 5
    xs = rng.standard_normal((T, hidden))
    w = rng.standard_normal((hidden, kernel_size))
    outs, buf = run_steps(xs, np.zeros((d_conv, hidden)), w)
    for ch in range(hidden):
        taps = w[ch, :d_conv + 1][::-1]  # convolve's h[m] weighs x[t - m]
        ref = np.convolve(xs[:, ch], taps)[:T]
        np.testing.assert_allclose(outs[:, ch], ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(buf, xs[T - d_conv:] if d_conv else np.zeros((0, hidden)))


def test_buffer_acts_as_earlier_inputs():
    rng = np.random.default_rng(2)
    d_conv, hidden = 3, 4
    w = rng.standard_normal((hidden, 4))
    pre = rng.standard_normal((d_conv, hidden))
    xs = rng.standard_normal((6, hidden))
    outs_a, buf_a = run_steps(xs, pre.copy(), w)
    _, buf0 = run_steps(pre, np.zeros((d_conv, hidden)), w)
    np.testing.assert_array_equal(buf0, pre)
    outs_b, buf_b = run_steps(xs, buf0, w)
    np.testing.assert_array_equal(outs_a, outs_b)
    np.testing.assert_array_equal(buf_a, buf_b)


def test_linearity_and_unused_taps():
    rng = np.random.default_rng(3)
    B, dc, h, ks = 3, 2, 6, 5
    x1, x2 = rng.standard_normal((2, B, h))
    b1, b2 = rng.standard_normal((2, B, dc, h))
    w1, w2 = rng.standard_normal((2, h, ks))
    o1, n1 = conv1d.conv1d_step(x1, b1, w1)
    o2, n2 = conv1d.conv1d_step(x2, b2, w1)
    o, n = conv1d.conv1d_step(2 * x1 - 3 * x2, 2 * b1 - 3 * b2, w1)
    np.testing.assert_allclose(o, 2 * o1 - 3 * o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(n, 2 * n1 - 3 * n2, rtol=1e-12, atol=1e-12)
    ow, _ = conv1d.conv1d_step(x1, b1, w1 + w2)
    np.testing.assert_allclose(ow, o1 + conv1d.conv1d_step(x1, b1, w2)[0], rtol=1e-12, atol=1e-12)
    w3 = w1.copy()
    w3[:, dc + 1:] = 1e9  # taps past d_conv
    np.testing.assert_array_equal(conv1d.conv1d_step(x1, b1, w3)[0], o1)


def test_batch_is_independent_sequences_and_inputs_untouched():
    rng = np.random.default_rng(4)
    B, dc, h = 4, 3, 7
    x = rng.standard_normal((B, h))
    buf = rng.standard_normal((B, dc, h))
    w = rng.standard_normal((h, dc + 1))
    keep = (x.copy(), buf.copy(), w.copy())
    o, n = conv1d.conv1d_step(x, buf, w)
    for b in range(B):
        ob, nb = conv1d.conv1d_step(x[b], buf[b], w)
        np.testing.assert_array_equal(o[b], ob)
        np.testing.assert_array_equal(n[b], nb)
    for a, k in zip((x, buf, w), keep):
        np.testing.assert_array_equal(a, k)


def test_kernel_size_too_small_is_refused():
    with pytest.raises(ValueError):
        conv1d.conv1d_step(np.zeros(3), np.zeros((2, 3)), np.zeros((3, 2)))
