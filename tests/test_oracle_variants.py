"""Pins of the oracle's ablation variants (AirCache notes, section "Ablation
studies": the observation-window table and the layer-budget table).

The page names the variants without formulas; the readings (R14, R15 in the
oracle's header) are checked here against closed forms and invariants that
any correct implementation of those readings satisfies."""
import numpy as np
import pytest

from oracle import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore")


# ------------------------------------------------------------------ windows

@pytest.mark.parametrize("n_t,mode,expect", [
    (5, 1, [0, 1, 2, 3, 4]),                # fewer text tokens than the window
    (40, 1, list(range(24, 40))),           # last 16
    (40, 2, list(range(8, 40))),            # last 32
    (16, 1, list(range(16))),               # exactly 16
    (7, 3, list(range(7))),                 # every text token
    (1, 2, [0]),
])
def test_window_positions(n_t, mode, expect):
    assert O.window(n_t, mode).tolist() == expect


@pytest.mark.parametrize("mode", [0, 4, -1])
def test_window_rejects_unknown_modes(mode):
    with pytest.raises(ValueError):
        O.window(10, mode)


# ------------------------------------------------------------------ budgets

def _layers(L, seed=0):
    rng = np.random.default_rng(seed)
    return rng.uniform(0.5, 2.0, L), rng.normal(1.0, 0.8, L)


def test_budget_mode_zero_is_the_method():
    st, sk = _layers(9)
    rl0, k0 = O.budget(st, sk, 5000, 0.1)
    rl, k = O.budget_variant(st, sk, 5000, 0.1, 0)
    assert np.array_equal(rl0, rl) and np.array_equal(k0, k)


@pytest.mark.parametrize("n_v,r", [(7290, 0.1), (1000, 0.25), (3, 1.0), (64, 0.01)])
def test_uniform_budget(n_v, r):
    st, sk = _layers(6, 1)
    rl, keep = O.budget_variant(st, sk, n_v, r, 1)
    assert np.all(rl == r)
    expect = min(max(int(np.floor(r * n_v + 0.5)), 1), n_v)
    assert np.all(keep == expect)


def test_pyramid_budget_closed_form():
    L, r = 5, 0.1
    st, sk = _layers(L, 2)
    rl, keep = O.budget_variant(st, sk, 2000, r, 2)
    # beta = 20: from (2 - 1/20) r at layer 0 to r / 20 at the last, linearly
    assert rl[0] == pytest.approx(1.95 * r, rel=1e-15)
    assert rl[-1] == pytest.approx(0.05 * r, rel=1e-15)
    assert np.allclose(np.diff(rl, 2), 0.0, atol=1e-15)
    assert np.mean(rl) == pytest.approx(r, rel=1e-14)
    assert keep.tolist() == [int(np.floor(x * 2000 + 0.5)) for x in rl]
    # it does not look at the statistics
    rl2, _ = O.budget_variant(st * 7.0, sk - 3.0, 2000, r, 2)
    assert np.array_equal(rl, rl2)


def test_pyramid_single_layer_is_uniform():
    rl, keep = O.budget_variant([1.0], [0.3], 100, 0.2, 2)
    assert rl.tolist() == [pytest.approx(0.2)] and keep.tolist() == [20]


def test_strength_only_budget():
    st = np.array([1.0, 2.0, 3.0, 6.0])
    sk = np.array([0.0, 5.0, -1.0, 2.0])
    rl, keep = O.budget_variant(st, sk, 1000, 0.1, 3)
    # s'_t = s_t / mean s_t (mean 3): r_l = r s_t / 3
    assert np.allclose(rl, 0.1 * st / 3.0, rtol=1e-15)
    assert keep.tolist() == [33, 67, 100, 200]
    # all-zero strengths give s'_t = 1
    rl0, _ = O.budget_variant(np.zeros(3), np.ones(3), 100, 0.3, 3)
    assert np.allclose(rl0, 0.3)


def test_skewness_only_budget():
    st = np.array([4.0, 1.0, 9.0])
    sk = np.array([0.5, 1.5, 1.0])
    rl, keep = O.budget_variant(st, sk, 1000, 0.1, 4)
    u = sk - 0.5 + 1e-6
    assert np.allclose(rl, 0.1 * u / u.mean(), rtol=1e-14)
    assert keep.tolist() == [1, 200, 100]  # the smallest skewness clamps to one token
    assert np.mean(rl) == pytest.approx(0.1, rel=1e-12)


@pytest.mark.parametrize("mode", [1, 2, 3, 4])
def test_variant_budgets_preserve_the_mean(mode):
    st, sk = _layers(11, 3)
    rl, _ = O.budget_variant(st, sk, 4000, 0.07, mode)
    assert np.mean(rl) == pytest.approx(0.07, rel=1e-12)


def test_budget_variant_rejects_unknown_modes():
    with pytest.raises(ValueError):
        O.budget_variant([1.0], [1.0], 10, 0.1, 5)


# ------------------------------------------------------------ whole request

def _request_inputs(seed=0, n_v=40, n_t=20, L=3, h_q=4, h_kv=2, d=8):
    rng = np.random.default_rng(seed)
    q = [(rng.standard_normal((n_t, h_q, d)) / np.sqrt(d)).astype(np.float32) for _ in range(L)]
    k = [rng.standard_normal((n_v + n_t, h_kv, d)).astype(np.float32) for _ in range(L)]
    return q, k, n_v


@pytest.mark.parametrize("window_mode", [1, 2, 3])
def test_request_with_a_window_scores_that_window(window_mode):
    q, k, n_v = _request_inputs(4)
    res = O.request(q, k, n_v, 0.9, 0.2, window_mode=window_mode)
    n_t = q[0].shape[0]
    win = O.window(n_t, window_mode)
    for l in range(len(q)):
        assert res["elite"][l].tolist() == win.tolist()
        iv, _ = O.score(q[l], k[l], n_v, win)
        assert np.array_equal(res["iv"][l], iv)


@pytest.mark.parametrize("budget_mode", [1, 2, 3, 4])
def test_request_with_a_budget_variant(budget_mode):
    q, k, n_v = _request_inputs(5)
    res = O.request(q, k, n_v, 0.9, 0.2, budget_mode=budget_mode)
    st, sk = res["stats"][:, 0], res["stats"][:, 1]
    _, keep = O.budget_variant(st, sk, n_v, 0.2, budget_mode)
    assert np.array_equal(res["keep"], keep)
    for l in range(len(q)):
        assert res["idx"][l].tolist() == O.select(res["iv"][l], int(keep[l])).tolist()


def test_default_request_is_unchanged():
    q, k, n_v = _request_inputs(6)
    a = O.request(q, k, n_v, 0.9, 0.2)
    b = O.request(q, k, n_v, 0.9, 0.2, window_mode=0, budget_mode=0)
    assert np.array_equal(a["iv"], b["iv"]) and np.array_equal(a["keep"], b["keep"])
