"""Pins of the oracle's per-KV-head index sets (reading R19: the edge-device
compression page's group-wise top-k, one decision per KV group)."""
import numpy as np
import pytest

from oracle import oracle as O


def _unit(seed, n_v=30, n_t=12, h_q=8, h_kv=4, d=16):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((n_t, h_q, d)) / np.sqrt(d)).astype(np.float32)
    k = rng.standard_normal((n_v + n_t, h_kv, d)).astype(np.float32)
    return q, k


def test_head_mean_of_the_group_scores_is_the_layer_score():
    q, k = _unit(1)
    el = np.array([3, 7, 11], np.int32)
    iv, ivh = O.score_heads(q, k, 30, el)
    assert np.allclose(ivh.mean(0), iv, rtol=1e-13, atol=0)
    iv2, _ = O.score(q, k, 30, el)
    assert np.array_equal(iv, iv2)


def test_one_kv_head_gives_the_layer_score():
    q, k = _unit(2, h_q=4, h_kv=1)
    el = np.array([0, 5], np.int32)
    iv, ivh = O.score_heads(q, k, 30, el)
    assert np.array_equal(ivh[0], iv)


def test_each_head_scores_its_own_group():
    # MHA: query head 0 looks at visual key 5, head 1 at visual key 3
    n_v, n_t, d = 8, 2, 8
    q = np.zeros((n_t, 2, d), np.float32)
    q[:, 0, 0] = 6.0
    q[:, 1, 1] = 6.0
    k = np.zeros((n_v + n_t, 2, d), np.float32)
    k[5, 0, 0] = 6.0
    k[3, 1, 1] = 6.0
    iv, ivh = O.score_heads(q, k, n_v, np.array([0, 1], np.int32))
    assert int(np.argmax(ivh[0])) == 5 and int(np.argmax(ivh[1])) == 3
    assert O.select(ivh[0], 1).tolist() == [5] and O.select(ivh[1], 1).tolist() == [3]


def test_request_selects_per_head_with_the_layer_budget():
    rng = np.random.default_rng(3)
    q = [(rng.standard_normal((12, 8, 16)) / 4).astype(np.float32) for _ in range(3)]
    k = [rng.standard_normal((42, 4, 16)).astype(np.float32) for _ in range(3)]
    a = O.request(q, k, 30, 0.9, 0.3, per_head=True)
    b = O.request(q, k, 30, 0.9, 0.3)
    assert np.array_equal(a["keep"], b["keep"]) and np.array_equal(a["iv"], b["iv"])
    for l in range(3):
        assert np.allclose(a["iv_heads"][l].mean(0), a["iv"][l], rtol=1e-13, atol=0)
        for h in range(4):
            assert a["idx_heads"][l][h].tolist() == O.select(a["iv_heads"][l][h], int(a["keep"][l])).tolist()


def test_compact_heads_row_order_and_agreement():
    n_v, n_t, h_kv, d = 5, 2, 2, 4
    src = np.zeros((n_v + n_t, h_kv, d), np.float32)
    for r in range(n_v + n_t):
        for h in range(h_kv):
            src[r, h] = 10 * r + h
    out = O.compact_heads(src, n_v, n_t, [[1, 4], [0, 2]])
    assert out[:, 0, 0].tolist() == [10.0, 40.0, 50.0, 60.0]
    assert out[:, 1, 0].tolist() == [1.0, 21.0, 51.0, 61.0]
    # the same set in every head is the shared-set compaction
    same = O.compact_heads(src, n_v, n_t, [[1, 3], [1, 3]], n_p=0)
    assert np.array_equal(same, O.compact(src, n_v, n_t, np.array([1, 3], np.int32)))
