"""Pins of the fp64 FFN oracle: FFN(x) = max(0, x W_1 + b_1) W_2 + b_2
("003-Transformer" tutorial, feed-forward layer; "From RNN to Attention", part 3)."""
import numpy as np
import torch

import oracle
from oracle import brute


def _w(d_model, d_ff, seed, bias=0.1):
    rng = np.random.default_rng(seed)
    return (rng.uniform(-0.2, 0.2, (d_ff, d_model)), rng.uniform(-bias, bias, d_ff),
            rng.uniform(-0.2, 0.2, (d_model, d_ff)), rng.uniform(-bias, bias, d_model))


def test_ffn_matches_torch_linear_relu_linear():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 5, 16))
    w1, b1, w2, b2 = _w(16, 40, 2)
    t = lambda a: torch.from_numpy(a)
    ref = torch.nn.functional.linear(torch.relu(torch.nn.functional.linear(t(x), t(w1), t(b1))), t(w2), t(b2))
    np.testing.assert_allclose(oracle.ffn_forward(x, w1, b1, w2, b2), ref.numpy(), rtol=0, atol=1e-13)


def test_ffn_brute_force_tiny():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 3, 4))
    w1, b1, w2, b2 = _w(4, 8, 4)
    got = oracle.ffn_forward(x, w1, b1, w2, b2)
    ref = np.array([brute.ffn_forward(x[b].tolist(), w1.tolist(), b1.tolist(), w2.tolist(), b2.tolist())
                    for b in range(2)])
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


def test_ffn_relu_cuts_negative_hidden_units():
    """A hidden bias far below zero switches every unit off: the output is exactly b_2."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 16))
    w1, _, w2, b2 = _w(16, 32, 6)
    out = oracle.ffn_forward(x, w1, np.full(32, -1e6), w2, b2)
    assert np.all(out == b2)
    # and with W_1 = I, b_1 = 0, W_2 = I: FFN(x) = relu(x)
    eye = np.eye(16)
    np.testing.assert_array_equal(oracle.ffn_forward(x, eye, None, eye, None), np.maximum(x, 0))


def test_ffn_same_input_same_output():
    """d2l: the same MLP is applied at every position, so equal inputs give equal outputs."""
    rng = np.random.default_rng(7)
    x = np.repeat(rng.standard_normal((1, 1, 16)), 5, axis=1)
    out = oracle.ffn_forward(x, *_w(16, 24, 8))
    for i in range(1, 5):
        np.testing.assert_array_equal(out[0, i], out[0, 0])
    assert out.shape == (1, 5, 16)
