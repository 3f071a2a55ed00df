"""Pins of the fp64 oracle against facts fixed by the AirCache notes and by
mathematics: hand-derived cases (tests/golden, each with its derivation),
closed forms, invariants, brute force on tiny inputs, and special cases that
reduce to a library routine.  CPU only."""
import itertools
import math

import numpy as np
import pytest

from conftest import golden

LN = math.log


def qk_arrays(n_t, h_q, h_kv, d, n_v):
    q = np.zeros((n_t, h_q, d), np.float32)
    k = np.zeros((n_v + n_t, h_kv, d), np.float32)
    return q, k


# ---------------------------------------------------------------- elite

def test_elite_single_head_hand(oracle):
    case = golden("elite_hand.json")["cases"][0]
    n_v, d = case["n_v"], case["d"]
    w = case["log_weights_head0"]
    n_t = len(w)
    q, k = qk_arrays(n_t, 1, 1, d, n_v)
    rng = np.random.default_rng(3)
    q[:] = rng.standard_normal(q.shape)           # earlier text rows: noise
    q[n_t - 1, 0] = [2.0, 0, 0, 0]                # the last text query
    k[:n_v] = rng.standard_normal((n_v, 1, d))
    for j, lw in enumerate(w):
        k[n_v + j, 0] = [lw, 0, 0, 0]
    el, P = oracle.elite(q, k, n_v, case["alpha"])
    np.testing.assert_allclose(P, case["expected_P"], rtol=1e-6)
    assert el.tolist() == case["expected_elite"]


def test_elite_mean_of_softmax_rows(oracle):
    case = golden("elite_hand.json")["cases"][1]
    n_v, d = case["n_v"], case["d"]
    q, k = qk_arrays(3, 2, 1, d, n_v)
    s2 = math.sqrt(2.0)
    q[2, 0] = [s2, 0]
    q[2, 1] = [0, s2]
    q[0:2] = 7.0  # not the last row
    k[n_v + 0, 0] = [LN(9), 0]
    k[n_v + 1, 0] = [0, LN(2)]
    k[n_v + 2, 0] = [0, 0]
    el, P = oracle.elite(q, k, n_v, 0.5)
    np.testing.assert_allclose(P, case["expected_P"], rtol=1e-6)
    assert el.tolist() == case["expected_elite_alpha_0.5"]
    el, _ = oracle.elite(q, k, n_v, 0.6)
    assert el.tolist() == case["expected_elite_alpha_0.6"]


def test_elite_gqa_head_map(oracle):
    case = golden("elite_hand.json")["cases"][2]
    n_v = case["n_v"]
    q, k = qk_arrays(3, 4, 2, 2, n_v)
    s2 = math.sqrt(2.0)
    q[2, 0] = q[2, 1] = [s2, 0]
    q[2, 2] = q[2, 3] = [0, s2]
    k[n_v + 0, 0] = [LN(9), 0]
    k[n_v + 1, 1] = [0, LN(4)]
    _, P = oracle.elite(q, k, n_v, 0.9)
    np.testing.assert_allclose(P, case["expected_P"], rtol=1e-6)


def rand_qk(seed, n_t=12, h_q=4, h_kv=2, d=16, n_v=20, scale=1.0):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((n_t, h_q, d)) * scale).astype(np.float32)
    k = (rng.standard_normal((n_v + n_t, h_kv, d)) * scale).astype(np.float32)
    return q, k


@pytest.mark.parametrize("seed", range(5))
def test_elite_alpha_limits(oracle, seed):
    q, k = rand_qk(seed)
    n_v = 20
    el0, P = oracle.elite(q, k, n_v, 0.0)
    assert el0.tolist() == list(range(12))               # alpha = 0: every text token
    el1, _ = oracle.elite(q, k, n_v, 1.0)
    assert el1.tolist() == [int(np.argmax(P))]           # alpha = 1: the maximum
    el9, _ = oracle.elite(q, k, n_v, 0.9)
    assert int(np.argmax(P)) in el9.tolist()             # argmax is always elite
    assert abs(P.sum() - 1.0) < 1e-12                    # mean of distributions
    assert all(P[j] >= 0.9 * P.max() for j in el9)
    assert all(P[j] < 0.9 * P.max() for j in set(range(12)) - set(el9.tolist()))


def test_elite_tied_maxima_inclusive(oracle):
    q, k = qk_arrays(4, 1, 1, 2, 3)
    q[3, 0] = [1.0, 0]
    for j, val in enumerate([1.0, 0.0, 1.0, -1.0]):
        k[3 + j, 0] = [val * math.sqrt(2.0), 0]
    el, _ = oracle.elite(q, k, 3, 1.0)
    assert el.tolist() == [0, 2]


def test_elite_parallel_key(oracle):
    """q_last parallel to one text key at large norm: that key alone is elite."""
    q, k = rand_qk(7, n_t=10, h_q=4, h_kv=4, d=8, n_v=5, scale=0.1)
    target = 6
    q[9] = 0.0
    for h in range(4):
        k[5 + target, h] = 0.0
        k[5 + target, h, h] = 30.0
        q[9, h, h] = 30.0
    el, _ = oracle.elite(q, k, 5, 0.9)
    assert el.tolist() == [target]


# ---------------------------------------------------------------- score

def test_score_hand_single_row(oracle):
    case = golden("score_hand.json")["cases"][0]
    q, k = qk_arrays(2, 1, 1, 1, 3)
    q[0, 0, 0] = -5.0
    q[1, 0, 0] = 1.0
    k[0:3, 0, 0] = [LN(1), LN(2), LN(3)]
    k[3, 0, 0] = LN(100)  # text 0, not elite
    k[4, 0, 0] = LN(4)    # text 1, elite
    iv, mass = oracle.score(q, k, 3, np.array([1]))
    np.testing.assert_allclose(iv, case["expected_iv"], rtol=1e-6)
    np.testing.assert_allclose(mass[0, 0], case["expected_mass"], rtol=1e-6)


def test_score_hand_rows_and_heads(oracle):
    case = golden("score_hand.json")["cases"][1]
    q, k = qk_arrays(2, 2, 1, 1, 2)
    q[0, 0, 0], q[0, 1, 0] = 1.0, 2.0
    q[1, 0, 0], q[1, 1, 0] = 0.0, -1.0
    k[0, 0, 0], k[1, 0, 0] = 0.0, LN(3)
    iv, _ = oracle.score(q, k, 2, np.array([0, 1]))
    np.testing.assert_allclose(iv, case["expected_iv"], rtol=1e-6)


@pytest.mark.parametrize("seed", range(4))
def test_score_mass_conservation(oracle, seed):
    q, k = rand_qk(seed, n_t=9, h_q=6, h_kv=3, d=8, n_v=30)
    el, _ = oracle.elite(q, k, 30, 0.5)
    iv, mass = oracle.score(q, k, 30, el)
    assert abs(iv.sum() + mass.mean() - 1.0) < 1e-12


def test_score_zero_queries_uniform(oracle):
    q, k = rand_qk(1, n_t=8, n_v=25)
    q[:] = 0.0
    el = np.array([1, 4, 6])
    iv, _ = oracle.score(q, k, 25, el)
    np.testing.assert_allclose(iv, 1.0 / (25 + 3), rtol=1e-14, atol=0)


def test_score_equal_visual_keys_constant(oracle):
    q, k = rand_qk(2, n_v=17)
    k[:17] = k[0]
    iv, _ = oracle.score(q, k, 17, np.array([0, 5]))
    assert np.ptp(iv) < 1e-15


def test_score_visual_permutation_equivariance(oracle):
    q, k = rand_qk(4, n_v=23)
    perm = np.random.default_rng(0).permutation(23)
    k2 = k.copy()
    k2[:23] = k[perm]
    el = np.array([2, 3, 11])
    iv, _ = oracle.score(q, k, 23, el)
    iv2, _ = oracle.score(q, k2, 23, el)
    np.testing.assert_allclose(iv2, iv[perm], rtol=1e-13, atol=0)


def test_score_matches_library_softmax(oracle):
    """A special case written with torch's fp64 softmax: for each head, the
    elite queries against [visual keys; elite text keys], column means."""
    import torch

    n_t, h_q, h_kv, d, n_v = 10, 6, 2, 16, 40
    q, k = rand_qk(9, n_t=n_t, h_q=h_q, h_kv=h_kv, d=d, n_v=n_v)
    el = np.array([0, 3, 7, 9])
    iv, _ = oracle.score(q, k, n_v, el)
    Q = torch.from_numpy(q).double()
    K = torch.from_numpy(k).double()
    g = h_q // h_kv
    cols = torch.cat([torch.arange(n_v), n_v + torch.from_numpy(el).long()])
    acc = torch.zeros(n_v, dtype=torch.float64)
    for h in range(h_q):
        A = torch.softmax(Q[el, h] @ K[cols, h // g].T / math.sqrt(d), dim=-1)
        acc += A[:, :n_v].mean(dim=0)
    np.testing.assert_allclose(iv, (acc / h_q).numpy(), rtol=1e-12, atol=1e-15)


def test_score_bf16_decoding(oracle):
    """bf16 bits decode exactly: the same values as fp32 give the same I_v."""
    import torch

    q, k = rand_qk(5, n_v=12)
    qb = torch.from_numpy(q).bfloat16()
    kb = torch.from_numpy(k).bfloat16()
    q32, k32 = qb.float().numpy(), kb.float().numpy()
    q16 = qb.view(torch.int16).numpy().view(np.uint16)
    k16 = kb.view(torch.int16).numpy().view(np.uint16)
    el = np.array([1, 2])
    a, _ = oracle.score(q32, k32, 12, el)
    b, _ = oracle.score(q16, k16, 12, el)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- stats

def test_stats_hand(oracle):
    for c in golden("stats_hand.json")["cases"]:
        s_t, s_k, mu, sigma = oracle.stats(np.array(c["iv"], dtype=np.float64))
        assert s_t == pytest.approx(c["s_t"], rel=1e-15)
        assert s_k == pytest.approx(c["s_k"], rel=1e-13, abs=1e-14), c


@pytest.mark.parametrize("n", [3, 5, 10, 64, 7290])
def test_skewness_one_hot_closed_form(oracle, n):
    x = np.zeros(n)
    x[n // 2] = 1.0
    assert oracle.stats(x)[1] == pytest.approx(math.sqrt(n), rel=1e-12)


def test_skewness_invariances(oracle):
    x = np.random.default_rng(0).exponential(size=101)
    s = oracle.stats(x)[1]
    assert oracle.stats(3.5 * x + 2.0)[1] == pytest.approx(s, rel=1e-12)
    assert oracle.stats(-x)[1] == pytest.approx(-s, rel=1e-12)


def test_skewness_matches_scipy(oracle):
    stats = pytest.importorskip("scipy.stats")
    for seed in range(5):
        x = np.random.default_rng(seed).gamma(0.5, size=500)
        assert oracle.stats(x)[1] == pytest.approx(stats.skew(x, bias=False), rel=1e-12)


def test_stats_rejects_short(oracle):
    with pytest.raises(ValueError):
        oracle.stats(np.array([1.0, 2.0]))


# ---------------------------------------------------------------- budget

def test_budget_hand(oracle):
    for c in golden("budget_hand.json")["cases"]:
        rl, keep = oracle.budget(c["s_t"], c["s_k"], c["n_v"], c["r"])
        np.testing.assert_allclose(rl, c["expected_r_l"], rtol=1e-12)
        assert keep.tolist() == c["expected_keep"], c["name"]


@pytest.mark.parametrize("seed", range(6))
def test_budget_preserves_mean(oracle, seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 40))
    s_t = rng.uniform(0.2, 1.0, L)
    s_k = rng.normal(3.0, 2.0, L)
    r = float(rng.uniform(0.01, 0.5))
    rl, keep = oracle.budget(s_t, s_k, 5000, r)
    assert abs(rl.mean() - r) < 1e-12
    assert np.all(keep >= 1) and np.all(keep <= 5000)
    # the arena bound used by the library: sum keep <= ceil(r L N_v) + 2L
    assert keep.sum() <= math.ceil(r * L * 5000) + 2 * L
    if L == 1:
        assert rl[0] == pytest.approx(r, rel=1e-15)


def test_budget_identical_layers(oracle):
    rl, keep = oracle.budget([0.3] * 5, [1.7] * 5, 7290, 0.1)
    np.testing.assert_allclose(rl, 0.1, rtol=1e-12)
    assert keep.tolist() == [729] * 5


# ---------------------------------------------------------------- select

@pytest.mark.parametrize("seed", range(20))
def test_select_brute_force(oracle, seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 13))
    iv = rng.random(n)
    kk = int(rng.integers(0, n + 1))
    best = max(itertools.combinations(range(n), kk), key=lambda s: sum(iv[list(s)]))
    assert oracle.select(iv, kk).tolist() == sorted(best)


def test_select_ties_lower_index(oracle):
    assert oracle.select(np.full(9, 0.25), 4).tolist() == [0, 1, 2, 3]
    assert oracle.select(np.array([5.0, 3, 3, 3, 1]), 2).tolist() == [0, 1]
    assert oracle.select(np.array([1.0, 3, 2, 3, 3]), 2).tolist() == [1, 3]
    assert oracle.select(np.array([0.0, 0, 0, 1e-300]), 2).tolist() == [0, 3]


# ---------------------------------------------------------------- compact

def test_compact_hand(oracle):
    src = np.arange(6 * 2 * 4, dtype=np.float32).reshape(6, 2, 4)  # N_v=4, N_t=2
    out = oracle.compact(src, 4, 2, np.array([1, 3]))
    assert np.array_equal(out, src[[1, 3, 4, 5]])


def test_compact_keep_all_is_identity(oracle):
    src = np.random.default_rng(0).integers(0, 65535, (30, 3, 8)).astype(np.uint16)
    out = oracle.compact(src, 26, 4, np.arange(26))
    assert np.array_equal(out, src)


def test_compact_strided_source(oracle):
    big = np.random.default_rng(1).standard_normal((10, 4, 8)).astype(np.float32)
    view = big[:, 1:3, :]                   # head-strided view
    out = oracle.compact(view, 7, 3, np.array([0, 6]))
    assert np.array_equal(out, view[[0, 6, 7, 8, 9]])


# ---------------------------------------------------------------- request

def test_request_heavy_keys_survive(oracle):
    """One layer, so r_l = r: the keep count is round(r N_v) and a handful of
    keys aligned with every elite query are the ones kept."""
    rng = np.random.default_rng(11)
    n_t, h_q, h_kv, d, n_v = 6, 4, 2, 16, 50
    q = rng.standard_normal((n_t, h_q, d)).astype(np.float32) * 0.3
    k = rng.standard_normal((n_v + n_t, h_kv, d)).astype(np.float32) * 0.3
    u = np.ones(d, np.float32) / math.sqrt(d)
    q += 2.0 * u
    heavy = [3, 17, 41]
    k[heavy] += 6.0 * u
    res = oracle.request([q], [k], n_v, 0.9, 0.06)
    assert res["keep"].tolist() == [3]
    assert res["idx"][0].tolist() == heavy
