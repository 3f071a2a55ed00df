"""Pins of the oracle's visual span at an offset (reading R18: the prompt is
[prefix text][visual][suffix text]; text is every non-visual token, prefix
then suffix; the multimodal-layout page puts the system text before the
visual tokens).

The layout moves rows, not arithmetic: the same tokens laid out visual-first
(n_p = 0, text in the same order) must give the same result, bit for bit."""
import numpy as np
import pytest

from oracle import oracle as O


def _request(seed, n_v=40, n_t=20, L=3, h_q=4, h_kv=2, d=8):
    rng = np.random.default_rng(seed)
    q = [(rng.standard_normal((n_t, h_q, d)) / np.sqrt(d)).astype(np.float32) for _ in range(L)]
    k_vis_first = [rng.standard_normal((n_v + n_t, h_kv, d)).astype(np.float32) for _ in range(L)]
    return q, k_vis_first


def _to_prefix(k, n_v, n_p):
    """Visual-first rows [visual; text] -> prompt order [text[:n_p]; visual; text[n_p:]]."""
    return np.concatenate([k[n_v:n_v + n_p], k[:n_v], k[n_v + n_p:]])


@pytest.mark.parametrize("n_p", [1, 7, 19, 20])
def test_prefix_layout_equals_visual_first(n_p):
    n_v = 40
    q, kv = _request(n_p)
    kp = [_to_prefix(k, n_v, n_p) for k in kv]
    a = O.request(q, kv, n_v, 0.9, 0.25)
    b = O.request(q, kp, n_v, 0.9, 0.25, n_p=n_p)
    assert np.array_equal(a["iv"], b["iv"]) and np.array_equal(a["keep"], b["keep"])
    for l in range(3):
        assert np.array_equal(a["elite"][l], b["elite"][l]) and np.array_equal(a["idx"][l], b["idx"][l])
        ca = O.compact(kv[l], n_v, 20, a["idx"][l])
        cb = O.compact(kp[l], n_v, 20, b["idx"][l], n_p=n_p)
        assert np.array_equal(ca, cb)


def test_prefix_layout_differs_from_reading_it_visual_first():
    # the same prompt-order rows read with n_p = 0 are a different problem
    n_v, n_p = 40, 7
    q, kv = _request(3)
    kp = [_to_prefix(k, n_v, n_p) for k in kv]
    b = O.request(q, kp, n_v, 0.9, 0.25, n_p=n_p)
    c = O.request(q, kp, n_v, 0.9, 0.25, n_p=0)
    assert not np.array_equal(b["iv"], c["iv"])


def test_a_prefix_token_can_be_elite():
    # the last query aligned with prefix key 2: the elite set is {2}
    n_v, n_t, n_p, d = 10, 6, 3, 8
    q = np.zeros((n_t, 1, d), np.float32)
    q[-1, 0, 0] = 10.0
    k = np.zeros((n_v + n_t, 1, d), np.float32)
    k[2, 0, 0] = 10.0          # prompt row 2 = text index 2 (in the prefix)
    k[n_p + 4, 0, 0] = 10.0    # visual index 4: not a text key
    el, P = O.elite(q, k, n_v, 0.9, n_p=n_p)
    assert el.tolist() == [2]
    assert P[2] == pytest.approx(1.0 / (1.0 + (n_t - 1) * np.exp(-100.0 / np.sqrt(d))))


def test_compact_row_order_with_prefix():
    # kept visual rows first, then the text rows in text order (prefix, suffix)
    n_v, n_t, n_p = 4, 3, 2
    rows = np.arange(n_v + n_t, dtype=np.float32).reshape(-1, 1, 1) * np.ones((1, 1, 8), np.float32)
    out = O.compact(rows, n_v, n_t, np.array([1, 3], np.int32), n_p=n_p)
    # prompt rows: 0,1 prefix text; 2..5 visual; 6 suffix text
    assert out[:, 0, 0].tolist() == [3.0, 5.0, 0.0, 1.0, 6.0]


def test_rejects_bad_prefix():
    q, kv = _request(4)
    with pytest.raises(ValueError):
        O.request(q, kv, 40, 0.9, 0.25, n_p=21)
    with pytest.raises(ValueError):
        O.elite(q[0], kv[0], 40, 0.9, n_p=-1)
