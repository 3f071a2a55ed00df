"""Pins of the oracle's visual observation window (reading R14: the ablation
table's visual window of 32 is the last 32 visual tokens; their queries attend
over the visual keys only)."""
import numpy as np
import pytest

from oracle import oracle as O


def test_window_is_the_last_32_visual_tokens():
    assert O.window_visual(100).tolist() == list(range(68, 100))
    assert O.window_visual(5).tolist() == [0, 1, 2, 3, 4]


def test_one_query_one_head_is_its_softmax_row():
    # one window row, one head: I_v is exactly that row's softmax over the visual keys
    rng = np.random.default_rng(1)
    n_v, n_t, d = 6, 3, 8
    qv = rng.standard_normal((n_v, 1, d)).astype(np.float32)
    k = rng.standard_normal((n_v + n_t, 1, d)).astype(np.float32)
    iv = O.score_visual_window(qv, k, n_v, [4])
    x = k[:n_v, 0].astype(np.float64) @ qv[4, 0].astype(np.float64) / np.sqrt(d)
    p = np.exp(x - x.max())
    assert np.allclose(iv, p / p.sum(), rtol=1e-14, atol=0)
    assert iv.sum() == pytest.approx(1.0, abs=1e-14)  # no text keys: every row's mass stays visual


def test_text_keys_do_not_enter():
    rng = np.random.default_rng(2)
    n_v, n_t = 10, 4
    qv = rng.standard_normal((n_v, 2, 8)).astype(np.float32)
    k = rng.standard_normal((n_v + n_t, 2, 8)).astype(np.float32)
    a = O.score_visual_window(qv, k, n_v, O.window_visual(n_v))
    k2 = k.copy()
    k2[n_v:] *= 100.0  # only text rows change
    assert np.array_equal(a, O.score_visual_window(qv, k2, n_v, O.window_visual(n_v)))
    # and with a prefix the visual rows move, the result does not
    n_p = 3
    kp = np.concatenate([k[n_v:n_v + n_p], k[:n_v], k[n_v + n_p:]])
    assert np.array_equal(a, O.score_visual_window(qv, kp, n_v, O.window_visual(n_v), n_p=n_p))


def test_request_with_the_visual_window():
    rng = np.random.default_rng(3)
    L, n_v, n_t = 2, 50, 12
    q = [rng.standard_normal((n_t, 4, 8)).astype(np.float32) for _ in range(L)]
    qv = [rng.standard_normal((n_v, 4, 8)).astype(np.float32) for _ in range(L)]
    k = [rng.standard_normal((n_v + n_t, 2, 8)).astype(np.float32) for _ in range(L)]
    res = O.request(q, k, n_v, 0.9, 0.2, window_mode=4, qv_layers=qv)
    for l in range(L):
        assert res["elite"][l].tolist() == list(range(18, 50))
        assert np.array_equal(res["iv"][l], O.score_visual_window(qv[l], k[l], n_v, O.window_visual(n_v)))
    with pytest.raises(ValueError):
        O.request(q, k, n_v, 0.9, 0.2, window_mode=4)  # the visual window needs the visual queries
