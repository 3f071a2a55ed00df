"""Comparison of the CUDA library's outputs with the fp64 oracle.

Acceptance rules (bf16/fp32 inputs, fp32 accumulation on the GPU):
  * elite sets equal, except positions whose fp64 head-mean weight P_j lies
    within 1e-5 * max P of the threshold alpha * max P (fp32 vs fp64 can flip
    those); where the sets differ, the oracle is re-run with the GPU's set;
  * I_v within 1e-3 relative / 1e-6 absolute;
  * (s_t, s_k) equal to the oracle's statistics of the GPU's I_v to 1e-9;
  * keep counts exactly equal to the oracle's budget applied to the GPU's I_v,
    and within one of the pure-oracle counts only where the oracle's r_l N_v
    lies within 1e-3 of a rounding boundary;
  * selection exactly equal to the oracle's selection on the GPU's I_v; against
    the oracle's own I_v the sets differ only by swaps whose I_v gap is within
    the I_v tolerance;
  * compaction bit-exact given the GPU's index set.
"""
from __future__ import annotations

import numpy as np

from lvlm_kv_cache_gb300 import workloads as W

IV_RTOL, IV_ATOL = 1e-3, 1e-6
ELITE_BAND = 1e-5


def unit_views(wl, l, b, cu_s, cu_v):
    """Host oracle views of one (layer, request): (q [N_t,H_q,D], k, v [N_v+N_t,H_kv,D])."""
    s0, s1 = cu_s[b], cu_s[b + 1]
    t0 = s0 - cu_v[b]
    n_t = (s1 - s0) - (cu_v[b + 1] - cu_v[b])
    q = W.host_bits(wl.q[l, t0:t0 + n_t])
    k = W.host_bits(wl.k[l, s0:s1])
    v = W.host_bits(wl.v[l, s0:s1])
    return q, k, v


def check_elite(oracle, q, k, n_v, alpha, gpu_elite):
    """Returns the oracle elite set to score with (the GPU's when they differ
    only inside the threshold band) and the number of band flips."""
    el, P = oracle.elite(q, k, n_v, alpha)
    g = np.asarray(gpu_elite, dtype=np.int64)
    if np.array_equal(el, g):
        return el, 0
    thr = alpha * P.max()
    diff = set(el.tolist()) ^ set(g.tolist())
    bad = [j for j in diff if abs(P[j] - thr) > ELITE_BAND * P.max()]
    assert not bad, f"elite sets differ outside the threshold band at {bad}: oracle {el} gpu {g}"
    return g.astype(np.int32), len(diff)


def check_iv(oracle_iv, gpu_iv, what=""):
    np.testing.assert_allclose(gpu_iv.astype(np.float64), oracle_iv, rtol=IV_RTOL, atol=IV_ATOL,
                               err_msg=f"I_v mismatch {what}")


def check_selection_vs_oracle_iv(oracle_iv, gpu_idx, keep):
    ref = np.sort(np.argsort(-oracle_iv, kind="stable")[:keep])
    gset, rset = set(gpu_idx.tolist()), set(ref.tolist())
    only_g, only_r = sorted(gset - rset), sorted(rset - gset)
    assert len(only_g) == len(only_r)
    if only_g:
        tol = IV_RTOL * np.abs(oracle_iv).max() + IV_ATOL
        assert oracle_iv[only_g].min() >= oracle_iv[only_r].max() - tol, "selection differs beyond swaps"
    return len(only_g)


def near_half(x, band=1e-3):
    f = x - np.floor(x)
    return abs(f - 0.5) < band


def check_unit(oracle, wl, l, b, cu_s, cu_v, gpu, report, window_mode=0):
    """Full per-(layer, request) check of elite (or the ablation window), I_v
    (stats/keep/select are checked per request by check_request)."""
    spec = wl.spec
    n_v = cu_v[b + 1] - cu_v[b]
    q, k, _ = unit_views(wl, l, b, cu_s, cu_v)
    u = l * spec.B + b
    ntk = int(gpu["n_tk"][u])
    g_el = gpu["elite"][u, :ntk]
    if window_mode:
        el = oracle.window(q.shape[0], window_mode)
        assert np.array_equal(g_el, el), f"window differs at (l={l}, b={b})"
    else:
        el, flips = check_elite(oracle, q, k, n_v, spec.alpha, g_el)
        report["elite_flips"] = report.get("elite_flips", 0) + flips
    iv_o, _ = oracle.score(q, k, n_v, el)
    iv_g = gpu["iv"][l, cu_v[b]:cu_v[b + 1]]
    check_iv(iv_o, iv_g, f"(l={l}, b={b})")
    report["max_rel_iv"] = max(report.get("max_rel_iv", 0.0),
                               float(np.max(np.abs(iv_g - iv_o) / (np.abs(iv_o) + IV_ATOL))))
    return iv_o


def check_request(oracle, wl, b, cu_s, cu_v, gpu, report, oracle_iv_by_layer=None, budget_mode=0):
    """Budget and selection of one request over all its layers, on the GPU's I_v."""
    spec = wl.spec
    n_v = cu_v[b + 1] - cu_v[b]
    st, sk = [], []
    for l in range(spec.L):
        iv_g = gpu["iv"][l, cu_v[b]:cu_v[b + 1]].astype(np.float64)
        s_t, s_k, _, _ = oracle.stats(iv_g)
        st.append(s_t)
        sk.append(s_k)
        if gpu.get("stats") is not None:
            u = l * spec.B + b
            np.testing.assert_allclose(gpu["stats"][u], [s_t, s_k], rtol=1e-9, atol=1e-12)
    rl, keep_o = oracle.budget_variant(st, sk, n_v, spec.r, budget_mode)
    keep_g = np.array([gpu["keep"][l * spec.B + b] for l in range(spec.L)])
    # distance of r_l * N_v from the nearest half-integer (where rounding turns)
    margin = [abs(rl[l] * n_v - np.floor(rl[l] * n_v) - 0.5) for l in range(spec.L)]
    report["half_margin"] = min(report.get("half_margin", np.inf), min(margin))
    boundary = [l for l in range(spec.L) if near_half(rl[l] * n_v, 1e-9)]
    mism = [l for l in range(spec.L) if keep_g[l] != keep_o[l] and l not in boundary]
    assert not mism, f"keep counts differ at layers {mism}: gpu {keep_g[mism]} oracle {keep_o[mism]}"
    # a mismatch inside the 1e-9 band is counted; strict callers fail on it
    report["near_half_exempt"] = report.get("near_half_exempt", 0) + sum(
        1 for l in boundary if keep_g[l] != keep_o[l])
    for l in range(spec.L):
        iv_g = gpu["iv"][l, cu_v[b]:cu_v[b + 1]].astype(np.float64)
        sel_o = oracle.select(iv_g, int(keep_g[l]))
        sel_g = gpu["idx"][l, cu_v[b]:cu_v[b] + int(keep_g[l])]
        assert np.array_equal(sel_o, sel_g), f"selection differs at l={l}, b={b}"
        if oracle_iv_by_layer is not None and l in oracle_iv_by_layer:
            report["swaps"] = report.get("swaps", 0) + check_selection_vs_oracle_iv(
                oracle_iv_by_layer[l], sel_g, int(keep_g[l]))
    if oracle_iv_by_layer is not None and len(oracle_iv_by_layer) == spec.L:
        st_o, sk_o = zip(*[oracle.stats(oracle_iv_by_layer[l])[:2] for l in range(spec.L)])
        rl_o, keep_oo = oracle.budget_variant(st_o, sk_o, n_v, spec.r, budget_mode)
        report["half_margin_oracle"] = min(report.get("half_margin_oracle", np.inf),
                                           min(abs(x * n_v - np.floor(x * n_v) - 0.5) for x in rl_o))
        for l in range(spec.L):
            if keep_oo[l] != keep_g[l]:
                assert abs(int(keep_oo[l]) - int(keep_g[l])) <= 1 and near_half(rl_o[l] * n_v), \
                    f"keep differs from the pure oracle at l={l}: {keep_g[l]} vs {keep_oo[l]}"
                report["keep_boundary"] = report.get("keep_boundary", 0) + 1
    return keep_g


def check_compaction(oracle, wl, l, b, cu_s, cu_v, gpu):
    spec = wl.spec
    u = l * spec.B + b
    n_v = cu_v[b + 1] - cu_v[b]
    n_t = (cu_s[b + 1] - cu_s[b]) - n_v
    kp = int(gpu["keep"][u])
    idx = gpu["idx"][l, cu_v[b]:cu_v[b] + kp]
    _, k, v = unit_views(wl, l, b, cu_s, cu_v)
    o0, o1 = int(gpu["out_offsets"][u]), int(gpu["out_offsets"][u + 1])
    assert o1 - o0 == kp + n_t
    exp_k = oracle.compact(k, n_v, n_t, idx)
    exp_v = oracle.compact(v, n_v, n_t, idx)
    assert np.array_equal(gpu["out_k"][o0:o1], exp_k), f"K rows differ at l={l}, b={b}"
    assert np.array_equal(gpu["out_v"][o0:o1], exp_v), f"V rows differ at l={l}, b={b}"


def expected_offsets(spec, keep):
    offs = [0]
    for l in range(spec.L):
        for b in range(spec.B):
            offs.append(offs[-1] + int(keep[l * spec.B + b]) + spec.n_text[b])
    return np.array(offs, dtype=np.int64)


def gpu_to_host(out, prob, n_tk=None, elite=None, stats=None):
    """Host copies of a compression's device outputs in oracle form."""
    res = {
        "iv": out["iv"].float().cpu().numpy(),
        "keep": out["keep"].cpu().numpy(),
        "idx": out["idx"].cpu().numpy(),
        "out_offsets": out["out_offsets"].cpu().numpy(),
    }
    rows = int(res["out_offsets"][-1])
    res["out_k"] = W.host_bits(out["out_k"][:rows])
    res["out_v"] = W.host_bits(out["out_v"][:rows])
    if n_tk is not None:
        res["n_tk"] = n_tk.cpu().numpy()
        res["elite"] = elite.cpu().numpy().reshape(prob.L * prob.B, -1)
    if stats is not None:
        res["stats"] = stats.cpu().numpy().reshape(prob.L * prob.B, 2)
    return res
