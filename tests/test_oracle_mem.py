"""Pins for the fp64 memory-combine oracle (oracle.mem_combine): attention of
each query over its retrieved memory (key, value) pairs, mixed with the local
output by a per-head weight.  Checked against closed forms and against the
already pinned band oracle, not against a second copy of its formula:

- weight 0 returns the local output exactly;
- one retrieved entry repeated in every slot returns its value row;
- q = 0 gives the plain mean of the retrieved value rows;
- every slot empty gives (1 - weight) * local;
- with the memory holding the sequence's own keys and values and the slots
  holding a row's window, the memory attention is the band oracle's output;
- a case worked out by hand; indices out of range are refused.
"""
import math

import numpy as np
import pytest

import oracle


def _rand(rng, B, H, n, d, M, km):
    q = rng.standard_normal((B, H, n, d))
    local = rng.standard_normal((B, H, n, d))
    mk = rng.standard_normal((B, H, M, d))
    mv = rng.standard_normal((B, H, M, d))
    idx = rng.integers(-1, M, size=(B, H, n, km)).astype(np.int32)
    return q, local, mk, mv, idx


def test_weight_zero_returns_local():
    rng = np.random.default_rng(1)
    q, local, mk, mv, idx = _rand(rng, 2, 3, 7, 8, 50, 32)
    out = oracle.mem_combine(q, local, mk, mv, idx, np.zeros(3))
    np.testing.assert_array_equal(out, local)


def test_repeated_entry_returns_its_value():
    rng = np.random.default_rng(2)
    q, local, mk, mv, _ = _rand(rng, 1, 2, 5, 4, 20, 8)
    idx = np.full((1, 2, 5, 8), 13, dtype=np.int32)
    out = oracle.mem_combine(q, local, mk, mv, idx, np.ones(2))
    for h in range(2):
        np.testing.assert_allclose(out[0, h], np.broadcast_to(mv[0, h, 13], (5, 4)), atol=1e-14, rtol=0)


def test_zero_query_gives_mean_of_retrieved_values():
    rng = np.random.default_rng(3)
    _, local, mk, mv, idx = _rand(rng, 2, 2, 6, 5, 30, 16)
    q = np.zeros((2, 2, 6, 5))
    out = oracle.mem_combine(q, local, mk, mv, idx, np.array([1.0, 0.25]))
    for b in range(2):
        for h in range(2):
            for i in range(6):
                sel = [j for j in idx[b, h, i] if j >= 0]
                om = mv[b, h, sel].mean(axis=0) if sel else np.zeros(5)
                g = [1.0, 0.25][h]
                np.testing.assert_allclose(out[b, h, i], g * om + (1 - g) * local[b, h, i], atol=1e-12, rtol=0)


def test_all_slots_empty_keeps_the_local_share():
    rng = np.random.default_rng(4)
    q, local, mk, mv, _ = _rand(rng, 1, 2, 4, 3, 10, 32)
    idx = np.full((1, 2, 4, 32), -1, dtype=np.int32)
    out = oracle.mem_combine(q, local, mk, mv, idx, np.array([0.3, 0.9]))
    np.testing.assert_allclose(out[0, 0], 0.7 * local[0, 0], atol=1e-15, rtol=0)
    np.testing.assert_allclose(out[0, 1], 0.1 * local[0, 1], atol=1e-15, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_memory_of_the_window_equals_the_band_attention(causal):
    rng = np.random.default_rng(5 + causal)
    B, H, n, d, w = 1, 2, 40, 8, 10
    q, k, v = (rng.standard_normal((B, H, n, d)) for _ in range(3))
    band = oracle.fwd(q, k, v, w=w, dilation=[1, 2], causal=causal)
    km = 32
    idx = np.full((B, H, n, km), -1, dtype=np.int32)
    for h in range(H):
        for i in range(n):
            keys, _ = oracle.attended(n=n, w=w, dilation=[1, 2], causal=causal, h=h, i=i)
            idx[0, h, i, :len(keys)] = keys
    out = oracle.mem_combine(q, np.zeros_like(q), k, v, idx, np.ones(H))
    np.testing.assert_allclose(out, band, atol=1e-12, rtol=0)


def test_case_worked_out_by_hand():
    """d = 1, q = ln 3: scores ln 3 and 0 against keys 1 and 0, weights 3/4 and
    1/4 over values 10 and 20: 12.5; with weight 1/2 and local 1: 6.75."""
    q = np.array([[[[math.log(3.0)]]]])
    mk = np.array([[[[1.0], [0.0]]]])
    mv = np.array([[[[10.0], [20.0]]]])
    idx = np.array([[[[0, 1]]]], dtype=np.int32)
    out = oracle.mem_combine(q, np.ones((1, 1, 1, 1)), mk, mv, idx, np.array([0.5]))
    assert abs(out[0, 0, 0, 0] - 6.75) <= 1e-12


def test_index_out_of_range_is_refused():
    rng = np.random.default_rng(6)
    q, local, mk, mv, idx = _rand(rng, 1, 1, 3, 2, 10, 4)
    idx[0, 0, 1, 2] = 10
    with pytest.raises(ValueError):
        oracle.mem_combine(q, local, mk, mv, idx, np.ones(1))
