"""Pins for the fp64 projection oracle (oracle.proj): per-head linear
projections of hidden states, y[t, b, h, i, c] = x[b, i] . w[t*H*d + h*d + c]
+ bias, checked against closed forms rather than against a second matmul:

- identity weights split the hidden state into heads exactly;
- a one-hot hidden state picks one column of the stacked weights, which fixes
  the order of the outputs t, the heads h and the columns c;
- zero input gives the bias; the map is additive and homogeneous;
- a product worked out by hand (tests/golden/proj_by_hand.json);
- bf16 inputs decode exactly.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_identity_weights_split_heads():
    rng = np.random.default_rng(1)
    B, n, H, d = 2, 5, 3, 4
    K = H * d
    x = rng.standard_normal((B, n, K))
    w = np.concatenate([np.eye(K), 2.0 * np.eye(K)])  # two outputs: x and 2x
    y = oracle.proj(x, w, H=H, d=d)
    assert y.shape == (2, B, H, n, d)
    for h in range(H):
        np.testing.assert_array_equal(y[0, :, h], x[:, :, h * d:(h + 1) * d])
        np.testing.assert_array_equal(y[1, :, h], 2.0 * x[:, :, h * d:(h + 1) * d])


def test_one_hot_input_picks_weight_columns():
    rng = np.random.default_rng(2)
    B, n, H, d, n_out, K = 1, 3, 2, 3, 3, 5
    w = rng.standard_normal((n_out * H * d, K))
    for kk in range(K):
        x = np.zeros((B, n, K))
        x[0, 1, kk] = 1.0
        y = oracle.proj(x, w, H=H, d=d)
        for t in range(n_out):
            for h in range(H):
                for c in range(d):
                    assert y[t, 0, h, 1, c] == w[t * H * d + h * d + c, kk]
        assert np.all(y[:, :, :, 0] == 0) and np.all(y[:, :, :, 2] == 0)


def test_zero_input_gives_bias_and_map_is_linear():
    rng = np.random.default_rng(3)
    B, n, H, d, K = 2, 4, 2, 8, 16
    w = rng.standard_normal((3 * H * d, K))
    bias = rng.standard_normal(3 * H * d).astype(np.float32)
    y0 = oracle.proj(np.zeros((B, n, K)), w, H=H, d=d, bias=bias)
    want = bias.astype(np.float64).reshape(3, 1, H, 1, d)
    np.testing.assert_array_equal(y0, np.broadcast_to(want, y0.shape))
    x1, x2 = rng.standard_normal((B, n, K)), rng.standard_normal((B, n, K))
    f = lambda x: oracle.proj(x, w, H=H, d=d)
    np.testing.assert_allclose(f(x1 + x2), f(x1) + f(x2), atol=1e-12, rtol=0)
    np.testing.assert_allclose(f(3.0 * x1), 3.0 * f(x1), atol=1e-12, rtol=0)


def test_product_worked_out_by_hand():
    case = json.load(open(os.path.join(GOLDEN, "proj_by_hand.json")))
    x = np.array(case["x"], dtype=np.float64)
    w = np.array(case["w"], dtype=np.float64)
    bias = np.array(case["bias"], dtype=np.float32)
    y = oracle.proj(x, w, H=case["H"], d=case["d"], bias=bias)
    np.testing.assert_array_equal(y, np.array(case["y"], dtype=np.float64))


def test_bf16_inputs_decode_exactly():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(2, 6, 32, generator=g).to(torch.bfloat16)
    w = torch.randn(3 * 2 * 16, 32, generator=g).to(torch.bfloat16)
    a = oracle.proj(x, w, H=2, d=16)
    b = oracle.proj(x.double(), w.double(), H=2, d=16)
    np.testing.assert_array_equal(a, b)


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.proj(np.zeros((1, 2, 4)), np.zeros((7, 4)), H=2, d=2)
