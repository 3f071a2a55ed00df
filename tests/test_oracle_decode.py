"""Pins of the oracle's decode step (reading R16: one query row attends over
every cached row; the KV-cache tutorial page, section "Prefill and Decode";
the edge-device compression page, head-wise top-k scheme, where decoding runs
dense attention over the compacted rows).

Each pin is a value fixed by the mathematics of softmax attention, not a
restatement of the oracle's loop."""
import math

import numpy as np
import pytest

from oracle import oracle as O


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


def test_single_row_returns_its_value_per_group():
    # one cached row: every weight is 1, so o_h is the value row of h's KV head
    h_q, h_kv, d = 6, 3, 8
    q = _rand((h_q, d), 1)
    k = _rand((1, h_kv, d), 2)
    v = _rand((1, h_kv, d), 3)
    out = O.decode(q, k, v)
    for h in range(h_q):
        assert np.array_equal(out[h], v[0, h // 2].astype(np.float64))


def test_zero_query_is_the_mean_of_the_values():
    # q = 0 makes every logit 0: uniform weights
    q = np.zeros((4, 16), np.float32)
    k = _rand((9, 2, 16), 4)
    v = _rand((9, 2, 16), 5)
    out = O.decode(q, k, v)
    for h in range(4):
        assert np.allclose(out[h], v[:, h // 2].astype(np.float64).mean(0), rtol=0, atol=1e-15)


def test_two_rows_closed_form():
    # D = 4, so the scale is 1/2; k1 . q / 2 = ln 3 makes the weights 1/4, 3/4
    d = 4
    q = np.zeros((1, d), np.float32)
    q[0, 0] = 1.0
    k = np.zeros((2, 1, d), np.float32)
    k[1, 0, 0] = np.float32(2.0 * math.log(3.0))
    v = np.zeros((2, 1, d), np.float32)
    v[0, 0] = [1.0, 0.0, -2.0, 4.0]
    v[1, 0] = [0.0, 8.0, 2.0, -4.0]
    logit1 = float(k[1, 0, 0]) / 2.0
    w1 = math.exp(logit1) / (1.0 + math.exp(logit1))
    expect = (1.0 - w1) * v[0, 0].astype(np.float64) + w1 * v[1, 0].astype(np.float64)
    out = O.decode(q, k, v)
    assert np.allclose(out[0], expect, rtol=0, atol=1e-15)
    assert w1 == pytest.approx(0.75, abs=1e-7)
    assert out[0, 1] == pytest.approx(6.0, abs=1e-6)


def test_dominant_row_takes_all_the_weight():
    d = 8
    q = np.zeros((2, d), np.float32)
    q[:, 0] = 40.0
    k = _rand((30, 1, d), 6) * 0.01
    k[17, 0, 0] = 40.0  # logit 40*40/sqrt(8) ~ 566 above the rest
    v = _rand((30, 1, d), 7)
    out = O.decode(q, k, v)
    assert np.allclose(out, np.broadcast_to(v[17, 0].astype(np.float64), (2, d)), rtol=0, atol=1e-12)
    assert np.isfinite(out).all()


def test_convex_combination_and_row_order():
    h_q, h_kv, d, n = 8, 2, 32, 50
    q = _rand((h_q, d), 8)
    k = _rand((n, h_kv, d), 9)
    v = _rand((n, h_kv, d), 10)
    out = O.decode(q, k, v)
    for h in range(h_q):
        vv = v[:, h // 4].astype(np.float64)
        assert np.all(out[h] <= vv.max(0) + 1e-12) and np.all(out[h] >= vv.min(0) - 1e-12)
    perm = np.random.default_rng(11).permutation(n)
    out_p = O.decode(q, k[perm], v[perm])
    assert np.allclose(out, out_p, rtol=0, atol=1e-13)


def test_strided_views_and_bf16():
    # a row of a wider arena, and bf16 storage (exact bit decode)
    h_kv, d = 2, 8
    arena = np.zeros((5, 3, d), np.uint16)  # 3 heads allocated, 2 used
    vals = np.array([0x3F80, 0x4000, 0xBF80, 0x3F00, 0x4040, 0x0000, 0x4080, 0xC000], np.uint16)  # 1,2,-1,.5,3,0,4,-2
    arena[2, 1] = vals
    k = arena[2:3, :h_kv]
    out = O.decode(np.ones((2, d), np.float32), k, arena[2:3, :h_kv])
    assert out[1].tolist() == [1.0, 2.0, -1.0, 0.5, 3.0, 0.0, 4.0, -2.0]
    assert out[0].tolist() == [0.0] * d


def test_compacted_cache_equals_the_same_rows_of_the_full_cache():
    # attention over the compacted rows (visual rows idx, then every text row)
    # is attention over that subset of the full cache
    n_v, n_t, h_q, h_kv, d = 40, 6, 4, 2, 16
    k = _rand((n_v + n_t, h_kv, d), 12)
    v = _rand((n_v + n_t, h_kv, d), 13)
    q = _rand((h_q, d), 14)
    idx = np.array([1, 5, 6, 20, 39], np.int32)
    ck = O.compact(k, n_v, n_t, idx)
    cv = O.compact(v, n_v, n_t, idx)
    rows = np.concatenate([idx, np.arange(n_v, n_v + n_t)])
    a = O.decode(q, ck, cv)
    b = O.decode(q, k[rows], v[rows])
    assert np.array_equal(a, b)


def test_rejects_empty_cache_and_bad_heads():
    with pytest.raises(ValueError):
        O.decode(np.zeros((2, 8), np.float32), np.zeros((0, 1, 8), np.float32), np.zeros((0, 1, 8), np.float32))
    with pytest.raises(ValueError):
        O.decode(np.zeros((3, 8), np.float32), np.zeros((2, 2, 8), np.float32), np.zeros((2, 2, 8), np.float32))
